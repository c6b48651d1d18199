"""Runs one decode step of a workload through the C ABI on the GPU and the
same step through the oracle on the CPU, and compares them."""
from contextlib import contextmanager

import numpy as np
import torch

import oracle
from oracle.block_table import BlockTable

TORCH = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16,
         "fp8_e4m3": torch.float8_e4m3fn}


def tolerance(cache_dtype):
    """(abs, rel) bound |gpu - ref| <= abs + rel * |ref| per element.
    fp16/bf16 caches: max-abs 2e-3 and rel 1e-2 in allclose form; fp8: max-abs
    5e-3 against the oracle on the same bytes and scales, plus one ulp of the
    16-bit output (2^-8 relative) — outputs are rounded to the q dtype, and a
    bf16 output above 1.28 in magnitude carries more than 5e-3 of rounding by
    itself; fp32: fp32 rounding of fp32 inputs (outputs ~1e-1)."""
    return {"f16": (2e-3, 1e-2), "bf16": (2e-3, 1e-2), "fp8_e4m3": (5e-3, 2.0 ** -8),
            "f32": (2e-5, 1e-4)}[cache_dtype]


def compare(got, ref, cache_dtype, what=""):
    got = got.detach().double().cpu().numpy() if isinstance(got, torch.Tensor) else got
    a, r = tolerance(cache_dtype)
    err = np.abs(got - ref)
    bound = a + r * np.abs(ref)
    stats = dict(max_abs=float(err.max()) if err.size else 0.0,
                 rel_l2=float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)))
    if not np.all(err <= bound):
        idx = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int((err > bound).sum())} elements out of tolerance; "
                             f"worst at {idx}: got {got[idx]!r} ref {ref[idx]!r}; {stats}")
    assert np.all(np.isfinite(got)), what
    return stats


def raw_bytes(t):
    t = t.detach().cpu().contiguous()
    return t.view(torch.uint8).numpy() if t.element_size() == 1 else t.view(torch.int16 if t.element_size() == 2 else torch.int32).numpy()


def run_gpu_step(w, num_splits=0, stream=None):
    """Returns (step, out) after adopt + append + attention on the GPU."""
    from paged_kv_gqa_03_gb300.step import DecodeStep
    dev = torch.device("cuda")
    stream = stream or torch.cuda.Stream()
    kc, vc = w.k_cache.to(dev), w.v_cache.to(dev)
    ks = None if w.k_scale is None else w.k_scale.to(dev)
    vs = None if w.v_scale is None else w.v_scale.to(dev)
    step = DecodeStep(kc, vc, w.Hq, TORCH[w.q_dtype], w.max_blocks, ks, vs,
                      num_splits=num_splits, stream=stream, scale=w.scale, q_len=w.q_len,
                      window=w.window)
    for b in range(w.B):
        step.adopt(b, w.tables[b], w.cached[b])
    step.prepare()
    step.upload()
    q, kn, vn = w.q.to(dev), w.k_new.to(dev), w.v_new.to(dev)
    out = torch.empty_like(q)
    step.launch(q, kn, vn, out)
    stream.synchronize()
    return step, out


def run_oracle_step(w):
    """The same step on the CPU: (slots, tables, lens, caches after append, out)."""
    bt = BlockTable(w.num_blocks)
    for b in range(w.B):
        bt.adopt(b, w.tables[b], w.cached[b])
    if w.window:
        for b in range(w.B):
            bt.release_outside_window(b, w.window)
    slots, cow = bt.append_slots([b for b in range(w.B) for _ in range(w.q_len)])
    assert cow == []
    mb = w.max_blocks
    table = np.full((w.B, mb), -1, dtype=np.int32)
    for b in range(w.B):
        t = bt.seq_tables[b]
        table[b, :len(t)] = t
    lens = np.array([bt.seq_tokens[b] for b in range(w.B)], dtype=np.int32)
    k_new = w.k_new.reshape(-1, w.Hkv, w.D)
    v_new = w.v_new.reshape(-1, w.Hkv, w.D)
    kc, vc, ks, vs = oracle.append(w.k_cache, w.v_cache, w.dtype, k_new, v_new, w.new_dtype,
                                   slots, None if w.k_scale is None else w.k_scale.numpy(),
                                   None if w.v_scale is None else w.v_scale.numpy())
    out = oracle.decode(w.q, w.q_dtype, kc, vc, w.dtype, table, lens, scale=w.scale,
                        k_scale=ks, v_scale=vs, window=w.window)
    return slots, table, lens, (kc, vc, ks, vs), out


@contextmanager
def routes(**choices):
    """Forces kernel-route decisions of the library (pkv_set_route) inside
    the block, e.g. routes(multi_query="transposed", prefill="tiles"), and
    restores the previous settings after it."""
    import paged_kv_gqa_03_gb300 as pkv
    prev = {k: pkv.pkv_set_route(k, v) for k, v in choices.items()}
    try:
        yield
    finally:
        for k, v in prev.items():
            pkv.pkv_set_route(k, v)
