"""GPU parity of the calibrated FP8 append (block scales follow the block's
running max as powers of two, earlier bytes re-quantised when it grows —
the calibration that "苦猿的大模型日记 Day45" PART 02 says decides FP8 quality):
caches and scales bit-exact against the oracle, and the attention error
against exact (unquantised) attention below that of the opener-only rule."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_helpers import compare

pytestmark = pytest.mark.gpu


def _pkv():
    import paged_kv_gqa_03_gb300 as pkv
    return pkv


def _stream(seed, B, Hkv, D, steps, per_call, new_dtype, start):
    """Token values whose magnitude drifts per token (lognormal factors), so
    blocks meet tokens larger than their first."""
    g = torch.Generator().manual_seed(seed)
    t = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[new_dtype]
    mag = torch.exp(torch.randn((steps, B, per_call, 1, 1), generator=g) * 0.7)
    x = torch.randn((steps, B, per_call, Hkv, D), generator=g) * mag
    y = torch.randn((steps, B, per_call, Hkv, D), generator=g) * mag
    return x.to(t), y.to(t)


@pytest.mark.parametrize("new_dtype,D,per_call", [("bf16", 128, 1), ("f16", 64, 1), ("f32", 128, 1),
                                                   ("bf16", 128, 5), ("bf16", 64, 3)])
def test_calibrated_append_is_bit_exact(new_dtype, D, per_call):
    """Six sequences append `per_call` tokens per call (consecutive entries,
    runs crossing block boundaries, sequences interleaved by call) for 12
    calls starting mid-block; caches and scales equal the oracle's after every
    call."""
    pkv = _pkv()
    dev = "cuda"
    B, Hkv, steps = 6, 2, 12
    start = [0, 5, 15, 16, 31, 40]
    nb = sum((s + steps * per_call + 15) // 16 for s in start) + 2
    g = torch.Generator().manual_seed(3)
    # blocks already holding `start` tokens, written by the plain rule
    kc = torch.randint(0, 0x7e, (nb, Hkv, 16, D), generator=g, dtype=torch.uint8)
    vc = kc.flip(-1).contiguous()
    ks = torch.rand((nb, Hkv), generator=g) * 0.01 + 0.001
    vs = torch.rand((nb, Hkv), generator=g) * 0.01 + 0.001
    perm = torch.randperm(nb, generator=g).tolist()
    tables, k = [], 0
    for s in start:
        n = (s + steps * per_call + 15) // 16
        tables.append(perm[k:k + n])
        k += n
    x, y = _stream(7, B, Hkv, D, steps, per_call, new_dtype, start)
    dk, dv, dks, dvs = kc.to(dev), vc.to(dev), ks.to(dev), vs.to(dev)
    rk, rv, rks, rvs = kc.numpy().copy(), vc.numpy().copy(), ks.numpy().copy(), vs.numpy().copy()
    pos = list(start)
    for it in range(steps):
        slots = []
        for b in range(B):
            for t in range(per_call):
                p = pos[b] + t
                slots.append(tables[b][p // 16] * 16 + p % 16)
            pos[b] += per_call
        kn = x[it].reshape(B * per_call, Hkv, D)
        vn = y[it].reshape(B * per_call, Hkv, D)
        pkv.paged_kv_append(kn.to(dev), vn.to(dev), dk.view(torch.float8_e4m3fn), dv.view(torch.float8_e4m3fn),
                            torch.tensor(slots, dtype=torch.int64, device=dev), dks, dvs, calibrated=True)
        rk, rv, rks, rvs = oracle.append(rk, rv, "fp8_e4m3", kn, vn, new_dtype, slots, k_scale=rks,
                                         v_scale=rvs, calibrated=True)
        torch.cuda.synchronize()
        assert np.array_equal(dk.cpu().numpy(), rk), f"K bytes, call {it}"
        assert np.array_equal(dv.cpu().numpy(), rv), f"V bytes, call {it}"
        assert np.array_equal(dks.cpu().numpy(), rks) and np.array_equal(dvs.cpu().numpy(), rvs), f"scales, call {it}"


def test_calibrated_decode_step_matches_oracle():
    """A whole decode step (append with calibration, then attention) on the
    long-context fp8 layer shape, reduced to 4 sequences."""
    w = workloads.config(5, B=4, ctx=[3000, 17, 33, 1500], free_frac=0.3, min_free=4)
    from paged_kv_gqa_03_gb300.step import DecodeStep
    dev = "cuda"
    stream = torch.cuda.Stream()
    step = DecodeStep(w.k_cache.to(dev), w.v_cache.to(dev), w.Hq, torch.bfloat16, w.max_blocks,
                      w.k_scale.to(dev), w.v_scale.to(dev), stream=stream, scale=w.scale, calibrated=True)
    for b in range(w.B):
        step.adopt(b, w.tables[b], w.cached[b])
    step.prepare()
    step.upload()
    out = torch.empty(w.q.shape, dtype=torch.bfloat16, device=dev)
    step.launch(w.q.to(dev), w.k_new.to(dev), w.v_new.to(dev), out)
    stream.synchronize()
    slots = step.h_slots.numpy()
    kc, vc, ks, vs = oracle.append(w.k_cache, w.v_cache, "fp8_e4m3", w.k_new, w.v_new, "bf16", slots,
                                   k_scale=w.k_scale.numpy(), v_scale=w.v_scale.numpy(), calibrated=True)
    assert np.array_equal(step.k_cache.cpu().view(torch.uint8).numpy(), kc)
    assert np.array_equal(step.k_scale.cpu().numpy(), ks)
    ref = oracle.decode(w.q, "bf16", kc, vc, "fp8_e4m3", step.h_table.numpy(), step.h_lens.numpy(),
                        scale=w.scale, k_scale=ks, v_scale=vs)
    compare(out, ref, "fp8_e4m3", "calibrated step")


def test_calibration_lowers_the_attention_error():
    """Sequences built token by token from a drifting-magnitude stream: the
    attention output over the calibrated FP8 cache is closer to exact
    attention over the unquantised values than over the opener-scaled cache."""
    pkv = _pkv()
    dev = "cuda"
    B, Hq, Hkv, D, T = 4, 8, 2, 128, 96
    nb = B * T // 16
    x, y = _stream(11, B, Hkv, D, T, 1, "bf16", [0] * B)
    q = torch.randn((B, Hq, D), generator=torch.Generator().manual_seed(2)).to(torch.bfloat16)
    table = torch.arange(nb, dtype=torch.int32).view(B, T // 16)
    lens = torch.full((B,), T, dtype=torch.int32)
    errs = {}
    for cal in (False, True):
        kc = torch.zeros((nb, Hkv, 16, D), dtype=torch.uint8, device=dev)
        vc = torch.zeros_like(kc)
        ks = torch.ones((nb, Hkv), device=dev)
        vs = torch.ones((nb, Hkv), device=dev)
        for t in range(T):
            slots = torch.tensor([b * T + t for b in range(B)], dtype=torch.int64, device=dev)
            pkv.paged_kv_append(x[t, :, 0].contiguous().to(dev), y[t, :, 0].contiguous().to(dev),
                                kc.view(torch.float8_e4m3fn), vc.view(torch.float8_e4m3fn), slots, ks, vs,
                                calibrated=cal)
        out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=dev)
        pkv.paged_decode_attention(out, q.to(dev), kc.view(torch.float8_e4m3fn), vc.view(torch.float8_e4m3fn),
                                   table.to(dev), lens.to(dev), 1 / math.sqrt(D), ks, vs)
        torch.cuda.synchronize()
        # exact attention over the unquantised values, laid out as an f32 cache
        kx = x[:, :, 0].float().permute(1, 0, 2, 3).reshape(nb, 16, Hkv, D).permute(0, 2, 1, 3).contiguous()
        vx = y[:, :, 0].float().permute(1, 0, 2, 3).reshape(nb, 16, Hkv, D).permute(0, 2, 1, 3).contiguous()
        ref = oracle.decode(q, "bf16", kx, vx, "f32", table.numpy(), lens.numpy(), scale=1 / math.sqrt(D))
        errs[cal] = float(np.sqrt(np.mean((out.double().cpu().numpy() - ref) ** 2)) / np.sqrt(np.mean(ref ** 2)))
    print("relative RMS error, opener-scaled vs calibrated:", errs)
    assert errs[True] < errs[False]


def test_mixed_precision_layers_share_one_block_table():
    """'大模型推理加速核心KV Cache 复用机制与内存布局优化' §四: keep FP16 KV in the
    key layers and FP8 elsewhere.  Three layers of one model step share the
    block manager's table, lengths and slot mapping; layers 0 and 2 use f16
    caches, layer 1 a calibrated fp8 cache; every layer's append and attention
    match the oracle."""
    pkv = _pkv()
    dev = "cuda"
    B, Hq, Hkv, D = 5, 16, 2, 128
    start = [33, 100, 7, 64, 250]
    nb = sum(s // 16 + 2 for s in start) + 4
    g = torch.Generator().manual_seed(17)
    bm = pkv.BlockManager(nb)
    for b, s in enumerate(start):
        assert bm.allocate(b, s)
    slots, pairs = bm.append_slots(list(range(B)))
    assert pairs == []
    table, lens = bm.export(list(range(B)), max(s // 16 + 2 for s in start))
    d_slots = torch.tensor(slots, dtype=torch.int64, device=dev)
    d_table, d_lens = torch.from_numpy(table).to(dev), torch.from_numpy(lens).to(dev)
    for layer, dtype in enumerate(("f16", "fp8_e4m3", "f16")):
        q = torch.randn((B, Hq, D), generator=g).to(torch.float16)
        kn = torch.randn((B, Hkv, D), generator=g).to(torch.float16)
        vn = torch.randn((B, Hkv, D), generator=g).to(torch.float16)
        if dtype == "f16":
            kc = torch.randn((nb, Hkv, 16, D), generator=g).to(torch.float16)
            vc = torch.randn((nb, Hkv, 16, D), generator=g).to(torch.float16)
            ks = vs = None
        else:
            kc = torch.randint(0, 0x7e, (nb, Hkv, 16, D), generator=g, dtype=torch.uint8).view(torch.float8_e4m3fn)
            vc = torch.randint(0, 0x7e, (nb, Hkv, 16, D), generator=g, dtype=torch.uint8).view(torch.float8_e4m3fn)
            ks = torch.rand((nb, Hkv), generator=g) * 0.01 + 0.001
            vs = torch.rand((nb, Hkv), generator=g) * 0.01 + 0.001
        dk, dv = kc.to(dev), vc.to(dev)
        dks = None if ks is None else ks.to(dev)
        dvs = None if vs is None else vs.to(dev)
        pkv.paged_kv_append(kn.to(dev), vn.to(dev), dk, dv, d_slots, dks, dvs, calibrated=True)
        out = torch.empty((B, Hq, D), dtype=torch.float16, device=dev)
        pkv.paged_decode_attention(out, q.to(dev), dk, dv, d_table, d_lens, 1 / math.sqrt(D), dks, dvs)
        torch.cuda.synchronize()
        rk, rv, rks, rvs = oracle.append(kc, vc, dtype, kn, vn, "f16", slots,
                                         None if ks is None else ks.numpy(), None if vs is None else vs.numpy(),
                                         calibrated=True)
        assert np.array_equal(dk.cpu().view(torch.uint8).numpy().reshape(-1), rk.view(np.uint8).reshape(-1))
        ref = oracle.decode(q, "f16", rk, rv, dtype, table, lens, scale=1 / math.sqrt(D), k_scale=rks,
                            v_scale=rvs)
        compare(out, ref, dtype, f"layer {layer} ({dtype})")
