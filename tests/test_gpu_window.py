"""GPU parity of sliding-window paged decode ("苦猿的大模型日记 Day45" PART 02:
a fixed visible history): each row attends its W most recent positions, the
kernel streams only the blocks inside the windows, and the block manager
releases blocks no later token can see.  Through the C ABI against the
oracle on the same seeded inputs."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_helpers import TORCH, compare, run_gpu_step, run_oracle_step

pytestmark = pytest.mark.gpu


def _pkv():
    import paged_kv_gqa_03_gb300 as pkv
    return pkv


def _bytes(t):
    return t.detach().cpu().contiguous().view(torch.uint8).numpy()


def _check_step(w, num_splits=0):
    step, out = run_gpu_step(w, num_splits=num_splits)
    slots, table, lens, (kc, vc, ks, vs), ref = run_oracle_step(w)
    assert step.h_slots.tolist() == slots
    assert np.array_equal(step.h_table.numpy(), table)       # released entries are -1 on both
    assert np.array_equal(step.h_lens.numpy(), lens)
    assert np.array_equal(_bytes(step.k_cache).reshape(-1), kc.view(np.uint8).reshape(-1))
    rc, flags = _pkv().paged_decode_status(step.workspace, step.stream)
    assert rc == 0 and flags == 0
    return compare(out, ref, w.dtype, f"{w.name} window {w.window} q_len {w.q_len}")


@pytest.mark.parametrize("spec", [
    dict(Hq=16, Hkv=2, D=128, dtype="bf16", window=1, ctx=[1, 17, 300]),
    dict(Hq=16, Hkv=2, D=128, dtype="bf16", window=16, ctx=[5, 16, 17, 33, 700]),
    dict(Hq=16, Hkv=2, D=128, dtype="bf16", window=17, ctx=[5, 16, 17, 33, 700]),
    dict(Hq=16, Hkv=2, D=64, dtype="bf16", window=100, ctx=[99, 100, 101, 1000]),
    dict(Hq=16, Hkv=2, D=128, dtype="bf16", window=37, q_len=4, ctx=[4, 40, 41, 600]),
    dict(Hq=8, Hkv=1, D=128, dtype="f16", window=50, q_len=3, ctx=[3, 52, 53, 257]),
    dict(Hq=8, Hkv=2, D=128, dtype="fp8_e4m3", q_dtype="bf16", window=45, ctx=[19, 46, 500]),
    dict(Hq=8, Hkv=2, D=64, dtype="fp8_e4m3", q_dtype="f16", window=20, q_len=2, ctx=[2, 40, 77]),
    dict(Hq=8, Hkv=2, D=128, dtype="f32", window=33, ctx=[3, 40, 177]),
    dict(Hq=2, Hkv=2, D=64, dtype="f32", window=9, q_len=2, ctx=[2, 18, 70]),
], ids=lambda s: f"{s['dtype']}-q{s['Hq']}-kv{s['Hkv']}-d{s['D']}-W{s['window']}-L{s.get('q_len', 1)}")
def test_window_shapes_and_dtypes(spec):
    """Windows of 1, of a block, of a block + 1 and beyond the context; q_len
    1-4 (each row its own window); partition counts 0, 5, 1000."""
    spec = dict(spec)
    spec.setdefault("q_dtype", spec["dtype"])
    spec["B"] = len(spec["ctx"])
    spec.update(free_frac=0.5, min_free=8)
    for seed, splits in ((5, 0), (6, 5), (7, 1000)):
        _check_step(workloads.make(spec, seed=seed), num_splits=splits)


@pytest.mark.parametrize("index,window", [(3, 4096), (5, 4096)])
def test_window_full_size(index, window):
    """The Llama-3.1-70B-shaped layer (64 x 8192, bf16) and the fp8 long-context
    layer (16 x 32768) with a 4096-position window, every output compared."""
    stats = _check_step(workloads.config(index, window=window))
    print(stats)


def test_window_steps_keep_the_cache_bounded():
    """Forty decode steps of 6 sequences with window 40 in a pool of only
    6 x 4 blocks (without releases the last steps would need 29): blocks
    released by the window are reused, and every step's output matches the
    oracle, which replays the same steps."""
    from oracle.block_table import BlockTable
    from paged_kv_gqa_03_gb300.step import DecodeStep
    dev = "cuda"
    B, Hq, Hkv, D, W, nb = 6, 16, 2, 128, 40, 24
    g = torch.Generator().manual_seed(23)
    kc = torch.randn((nb, Hkv, 16, D), generator=g).to(torch.bfloat16)
    vc = torch.randn((nb, Hkv, 16, D), generator=g).to(torch.bfloat16)
    step = DecodeStep(kc.to(dev), vc.to(dev), Hq, torch.bfloat16, 64, scale=0.088, window=W)
    ref_bt = BlockTable(nb)
    start = [1, 15, 16, 30, 47, 60]
    for b in range(B):
        assert step.bm.allocate(b, start[b]) and ref_bt.allocate(b, start[b])
        step.seqs.append(b)
    # the prompt positions hold the pool's random values already
    kr, vr = kc.clone(), vc.clone()
    for it in range(40):
        q = torch.randn((B, Hq, D), generator=g).to(torch.bfloat16)
        kn = torch.randn((B, Hkv, D), generator=g).to(torch.bfloat16)
        vn = torch.randn((B, Hkv, D), generator=g).to(torch.bfloat16)
        step.prepare()
        step.upload()
        out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=dev)
        step.launch(q.to(dev), kn.to(dev), vn.to(dev), out)
        step.stream.synchronize()
        for b in range(B):
            ref_bt.release_outside_window(b, W)
        slots, cow = ref_bt.append_slots(list(range(B)))
        assert cow == [] and step.h_slots.tolist() == slots
        kr, vr, _, _ = oracle.append(kr, vr, "bf16", kn, vn, "bf16", slots)
        table = np.full((B, 64), -1, dtype=np.int32)
        for b in range(B):
            table[b, :len(ref_bt.seq_tables[b])] = ref_bt.seq_tables[b]
        lens = np.array([ref_bt.seq_tokens[b] for b in range(B)], dtype=np.int32)
        assert np.array_equal(step.h_table.numpy(), table)
        ref = oracle.decode(q, "bf16", kr, vr, "bf16", table, lens, scale=0.088, window=W)
        compare(out, ref, "bf16", f"window step {it}")
        held = sum(int((table[b] >= 0).sum()) for b in range(B))
        assert held <= B * 4 and step.bm.num_free() == nb - held
