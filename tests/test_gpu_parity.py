"""GPU parity: every step of the decode path through the C ABI against the
oracle on the same seeded inputs.  Append and copy are compared bit for bit,
attention within the tolerances of gpu_helpers.tolerance."""
import math

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
    # a1: the native block manager agrees with the oracle's block table
    assert step.h_slots.tolist() == slots
    assert np.array_equal(step.h_table.numpy(), table)
    assert np.array_equal(step.h_lens.numpy(), lens)
    # a3: append is bit-exact (and writes nothing else)
    assert np.array_equal(_bytes(step.k_cache).reshape(-1), kc.view(np.uint8).reshape(-1))
    assert np.array_equal(_bytes(step.v_cache).reshape(-1), vc.view(np.uint8).reshape(-1))
    if ks is not None:
        assert np.array_equal(step.k_scale.cpu().numpy(), ks)
        assert np.array_equal(step.v_scale.cpu().numpy(), vs)
    # a4-a8: attention
    rc, flags = _pkv().paged_decode_status(step.workspace, step.stream)
    assert rc == 0 and flags == 0
    return compare(out, ref, w.dtype, w.name)


@pytest.mark.parametrize("index", [1, 2, 3, 4, 5])
def test_workload_full_size(index):
    """The five decode workloads at full size, every output compared."""
    w = workloads.config(index)
    stats = _check_step(w)
    print(f"workload {index}: {stats}")


@pytest.mark.parametrize("index,over", [
    (2, dict(B=5, ctx_range=(17, 300))),
    (3, dict(B=3, ctx=[1000, 17, 33], free_frac=0.3, min_free=3)),
    (4, dict(B=9, suffix_range=(1, 70))),
    (5, dict(B=2, ctx=[700, 33], free_frac=0.3, min_free=2)),
])
def test_workload_small(index, over):
    _check_step(workloads.config(index, **over))


@pytest.mark.parametrize("num_splits", [1, 2, 3, 8, 17, 1000, 0])
def test_result_independent_of_partition_count(num_splits):
    w = workloads.make(dict(B=6, Hq=16, Hkv=2, D=128, dtype="bf16", q_dtype="bf16",
                            ctx_range=(1, 600), free_frac=0.2), seed=77)
    _check_step(w, num_splits=num_splits)


@pytest.mark.parametrize("spec", [
    dict(B=7, Hq=8, Hkv=1, D=128, dtype="bf16", ctx=[1, 15, 16, 17, 32, 33, 48]),  # MQA, edges
    dict(B=3, Hq=16, Hkv=1, D=128, dtype="bf16", ctx=[40, 257, 5]),                 # group 16
    dict(B=3, Hq=6, Hkv=2, D=128, dtype="bf16", ctx=[40, 77, 5]),                   # group 3
    dict(B=3, Hq=4, Hkv=2, D=128, dtype="bf16", ctx=[40, 77, 5]),                   # group 2
    dict(B=3, Hq=4, Hkv=4, D=128, dtype="bf16", ctx=[40, 77, 5]),                   # MHA
    dict(B=3, Hq=8, Hkv=2, D=64, dtype="bf16", ctx=[40, 177, 5]),                   # D 64
    dict(B=3, Hq=8, Hkv=2, D=128, dtype="f16", ctx=[40, 177, 5]),                   # f16 MMA
    dict(B=3, Hq=8, Hkv=2, D=64, dtype="f16", ctx=[40, 177, 5]),
    dict(B=4, Hq=8, Hkv=8, D=128, dtype="f16", ctx=[40, 177, 5, 16]),               # f16 MHA
    dict(B=3, Hq=8, Hkv=2, D=128, dtype="fp8_e4m3", q_dtype="bf16", ctx=[40, 177, 17]),
    dict(B=3, Hq=8, Hkv=2, D=64, dtype="fp8_e4m3", q_dtype="bf16", ctx=[40, 177, 17]),
    dict(B=3, Hq=8, Hkv=2, D=128, dtype="fp8_e4m3", q_dtype="f16", ctx=[40, 177, 17]),
    dict(B=3, Hq=2, Hkv=2, D=128, dtype="fp8_e4m3", q_dtype="bf16", ctx=[40, 177, 17]),  # fp8 MHA
    dict(B=3, Hq=4, Hkv=2, D=64, dtype="fp8_e4m3", q_dtype="f16", ctx=[40, 177, 17]),    # fp8 group 2
    dict(B=3, Hq=8, Hkv=2, D=128, dtype="f32", ctx=[40, 177, 17]),
    dict(B=3, Hq=2, Hkv=1, D=64, dtype="f32", ctx=[40, 177, 17]),
    dict(B=2, Hq=8, Hkv=2, D=128, dtype="bf16", ctx=[17, 33], pool=12),             # block-opening appends
], ids=lambda s: f"{s['dtype']}-q{s['Hq']}-kv{s['Hkv']}-d{s['D']}")
def test_shapes_and_dtypes(spec):
    spec = dict(spec)
    spec.setdefault("q_dtype", spec["dtype"])
    spec.setdefault("free_frac", 0.5)
    spec.setdefault("min_free", 4)
    _check_step(workloads.make(spec, seed=5), num_splits=0)
    _check_step(workloads.make(spec, seed=6), num_splits=5)


def _attend(q, kc, vc, table, lens, scale, ks=None, vs=None, num_splits=0):
    pkv = _pkv()
    out = torch.empty_like(q)
    ws = pkv.paged_decode_attention(out, q, kc, vc, table, lens, scale, ks, vs, num_splits=num_splits)
    torch.cuda.synchronize()
    return out, ws


def test_closed_forms_and_empty_context():
    dev = "cuda"
    g = torch.Generator().manual_seed(3)
    Hq, Hkv, D, nb = 8, 2, 128, 8
    q = torch.randn((3, Hq, D), generator=g).to(torch.bfloat16)
    kc = torch.randn((nb, Hkv, 16, D), generator=g).to(torch.bfloat16)
    vc = torch.randn((nb, Hkv, 16, D), generator=g).to(torch.bfloat16)
    # seq 0: all keys equal -> mean of V; seq 1: a needle key = 50 q; seq 2: empty
    kc[0:2] = 0.25
    kc[2, 0, 3] = (50.0 * q[1, 0].float()).to(torch.bfloat16)
    table = torch.tensor([[0, 1], [2, 3], [4, 5]], dtype=torch.int32)
    lens = torch.tensor([20, 30, 0], dtype=torch.int32)
    out, ws = _attend(q.to(dev), kc.to(dev), vc.to(dev), table.to(dev), lens.to(dev), 1 / math.sqrt(D))
    got = out.double().cpu()
    mean_v = torch.cat([vc[0], vc[1]], dim=1)[:, :20].double().mean(dim=1)   # [Hkv, D]
    assert torch.allclose(got[0, :4], mean_v[0].expand(4, D), atol=2e-3, rtol=1e-2)
    assert torch.allclose(got[0, 4:], mean_v[1].expand(4, D), atol=2e-3, rtol=1e-2)
    assert torch.allclose(got[1, 0], vc[2, 0, 3].double(), atol=2e-3, rtol=1e-2)
    assert torch.all(got[2] == 0)
    ref = oracle.decode(q, "bf16", kc, vc, "bf16", table.numpy(), lens.numpy(), scale=1 / math.sqrt(D))
    compare(out, ref, "bf16", "closed forms")


def test_bad_block_id_and_length_are_flagged_not_faulted():
    pkv = _pkv()
    dev = "cuda"
    Hq, Hkv, D, nb = 8, 2, 128, 4
    q = torch.randn((2, Hq, D)).to(torch.bfloat16).to(dev)
    kc = torch.randn((nb, Hkv, 16, D)).to(torch.bfloat16).to(dev)
    vc = torch.randn((nb, Hkv, 16, D)).to(torch.bfloat16).to(dev)
    table = torch.tensor([[0, 99], [1, 2]], dtype=torch.int32, device=dev)
    lens = torch.tensor([20, 10], dtype=torch.int32, device=dev)
    out, ws = _attend(q, kc, vc, table, lens, 0.1)
    rc, flags = pkv.paged_decode_status(ws)
    assert rc == pkv.PKV_ERANGE and flags == 4
    assert torch.isfinite(out.float()).all()
    lens = torch.tensor([20, 10_000], dtype=torch.int32, device=dev)   # > 16 * max_blocks
    table = torch.tensor([[0, 3], [1, 2]], dtype=torch.int32, device=dev)
    out, ws = _attend(q, kc, vc, table, lens, 0.1)
    rc, flags = pkv.paged_decode_status(ws)
    assert rc == pkv.PKV_ERANGE and flags == 2
    ref = oracle.decode(q.cpu(), "bf16", kc.cpu(), vc.cpu(), "bf16", table.cpu().numpy(),
                        np.array([20, 32], dtype=np.int32), scale=0.1)
    compare(out, ref, "bf16", "clamped length")


def test_copy_on_write_append_into_shared_partial_block():
    """Prefix of 390 tokens (24 full blocks + 6 tokens) shared by a parent and
    two forks; both forks append, so each copies the shared partial block; the
    parent's cache and output are unchanged ("LLM推理优化实战" §2.2 CoW)."""
    pkv = _pkv()
    from paged_kv_gqa_03_gb300.step import DecodeStep
    from oracle.block_table import BlockTable
    dev = "cuda"
    Hq, Hkv, D, nb = 32, 8, 128, 40
    g = torch.Generator().manual_seed(9)
    kc = torch.randn((nb, Hkv, 16, D), generator=g).to(torch.bfloat16)
    vc = torch.randn((nb, Hkv, 16, D), generator=g).to(torch.bfloat16)
    q = torch.randn((3, Hq, D), generator=g).to(torch.bfloat16)
    kn = torch.randn((2, Hkv, D), generator=g).to(torch.bfloat16)
    vn = torch.randn((2, Hkv, D), generator=g).to(torch.bfloat16)
    step = DecodeStep(kc.to(dev), vc.to(dev), Hq, torch.bfloat16, 32)
    step.bm.allocate(0, 390)
    step.bm.fork(0, 1)
    step.bm.fork(0, 2)
    ref_bt = BlockTable(nb)
    ref_bt.allocate(0, 390)
    ref_bt.fork(0, 1)
    ref_bt.fork(0, 2)
    # parent's output before the forks write
    t0, l0 = step.bm.export([0], 32)
    out_parent_before, _ = _attend(q[:1].to(dev), step.k_cache, step.v_cache,
                                   torch.from_numpy(t0).to(dev), torch.from_numpy(l0).to(dev), 0.09,
                                   num_splits=1)
    ncow = step.prepare([1, 2])
    step.upload()
    assert ncow == 2
    slots_ref, cow_ref = ref_bt.append_slots([1, 2])
    assert step.h_slots.tolist() == slots_ref
    assert [tuple(step.h_pairs[2 * i:2 * i + 2].tolist()) for i in range(2)] == cow_ref
    step.launch(q[1:].to(dev), kn.to(dev), vn.to(dev), torch.empty((2, Hq, D), dtype=torch.bfloat16, device=dev))
    step.stream.synchronize()
    # oracle: copy then append on host copies
    kr, vr = kc.clone(), vc.clone()
    for src, dst in cow_ref:
        kr[dst], vr[dst] = kr[src], vr[src]
    kr, vr, _, _ = oracle.append(kr, vr, "bf16", kn, vn, "bf16", slots_ref)
    assert np.array_equal(_bytes(step.k_cache), kr.view(np.uint8).reshape(_bytes(step.k_cache).shape))
    assert np.array_equal(_bytes(step.v_cache), vr.view(np.uint8).reshape(_bytes(step.v_cache).shape))
    # all three sequences attend; the parent's result is bit-identical to before
    table, lens = step.bm.export([0, 1, 2], 32)
    out, _ = _attend(q.to(dev), step.k_cache, step.v_cache, torch.from_numpy(table).to(dev),
                     torch.from_numpy(lens).to(dev), 0.09, num_splits=1)
    assert torch.equal(out[:1], out_parent_before)   # one worker: same blocks, same order
    ref = oracle.decode(q, "bf16", kr, vr, "bf16", table, lens, scale=0.09)
    compare(out, ref, "bf16", "cow")


def test_append_skips_negative_slots_and_copy_blocks_is_exact():
    pkv = _pkv()
    dev = "cuda"
    for dtype in ("bf16", "fp8_e4m3"):
        g = torch.Generator().manual_seed(4)
        nb, Hkv, D = 6, 2, 128
        if dtype == "fp8_e4m3":
            kc = torch.randint(0, 0x7e, (nb, Hkv, 16, D), generator=g, dtype=torch.uint8).view(torch.float8_e4m3fn)
            ks = torch.rand((nb, Hkv), generator=g) * 0.01 + 0.001
        else:
            kc = torch.randn((nb, Hkv, 16, D), generator=g).to(torch.bfloat16)
            ks = None
        vc, vs = kc.clone(), (None if ks is None else ks.clone())
        new_t = torch.bfloat16
        kn = torch.randn((3, Hkv, D), generator=g).to(new_t)
        vn = torch.randn((3, Hkv, D), generator=g).to(new_t)
        slots = torch.tensor([2 * 16 + 5, -1, 4 * 16], dtype=torch.int64)
        dk, dv = kc.to(dev), vc.to(dev)
        dks = None if ks is None else ks.to(dev)
        dvs = None if vs is None else vs.to(dev)
        pkv.paged_kv_append(kn.to(dev), vn.to(dev), dk, dv, slots.to(dev), dks, dvs)
        kr, vr, ksr, vsr = oracle.append(kc, vc, dtype, kn, vn, "bf16", slots.numpy(),
                                         None if ks is None else ks.numpy(),
                                         None if vs is None else vs.numpy())
        torch.cuda.synchronize()
        assert np.array_equal(_bytes(dk), kr.view(np.uint8).reshape(_bytes(dk).shape))
        assert np.array_equal(_bytes(dv), vr.view(np.uint8).reshape(_bytes(dv).shape))
        if ks is not None:
            assert np.array_equal(dks.cpu().numpy(), ksr) and np.array_equal(dvs.cpu().numpy(), vsr)
        pairs = torch.tensor([[2, 0], [4, 5]], dtype=torch.int32, device=dev)
        pkv.paged_kv_copy_blocks(dk, dv, pairs, dks, dvs)
        torch.cuda.synchronize()
        k_host = dk.cpu()
        assert torch.equal(k_host[0].view(torch.uint8), k_host[2].view(torch.uint8))
        assert torch.equal(k_host[5].view(torch.uint8), k_host[4].view(torch.uint8))
        if ks is not None:
            assert torch.equal(dks[0], dks[2]) and torch.equal(dvs[5], dvs[4])


def test_exported_merge_matches_oracle():
    pkv = _pkv()
    g = torch.Generator().manual_seed(5)
    B, Hq, S, D = 3, 4, 5, 128
    o = torch.randn((B, Hq, S, D), generator=g)
    lse = torch.randn((B, Hq, S), generator=g) * 3
    lse[0, 0, 1:] = float("-inf")
    lse[1, 2, :] = float("-inf")
    for odt, name in ((torch.float32, "f32"), (torch.bfloat16, "bf16")):
        out = torch.empty((B, Hq, D), dtype=odt, device="cuda")
        pkv.paged_decode_merge(out, o.cuda(), lse.cuda())
        torch.cuda.synchronize()
        ref = oracle.merge(o.double().reshape(B * Hq, S, D).numpy(),
                           lse.double().reshape(B * Hq, S).numpy()).reshape(B, Hq, D)
        compare(out, ref, "f32" if name == "f32" else "bf16", "merge")


def test_captured_step_graph_matches_eager_step():
    """A whole step captured as a CUDA graph (copies, append, attention, copy
    back) gives the eager step's output bit for bit and the same caches."""
    w = workloads.config(3, B=4, ctx=[700, 17, 33, 1500], free_frac=0.3, min_free=4)
    step, out = run_gpu_step(w)
    eager_out = out.cpu()
    eager_k = step.k_cache.cpu()
    step.h_q.copy_(w.q)
    step.h_k_new.copy_(w.k_new)
    step.h_v_new.copy_(w.v_new)
    hout = torch.empty(w.q.shape, dtype=w.q.dtype).pin_memory()
    step.capture(hout)
    for _ in range(2):
        hout.zero_()
        step.replay()
        step.stream.synchronize()
        assert torch.equal(hout, eager_out)
    assert torch.equal(step.k_cache.cpu(), eager_k)


def test_large_batch_is_planned_by_the_plan_kernel():
    """Batches of 2048 sequences and more are planned by a separate kernel
    (smaller ones inside the decode kernel); both give the oracle's result and
    flag a bad context length."""
    spec = dict(B=2100, Hq=8, Hkv=2, D=64, dtype="bf16", ctx_range=(1, 40), free_frac=0.2, min_free=64)
    _check_step(workloads.make(spec, seed=21))
    pkv = _pkv()
    w = workloads.make(dict(spec, B=2050), seed=22)
    dev = "cuda"
    table = np.full((w.B, 3), 0, dtype=np.int32)
    for b in range(w.B):
        table[b, :len(w.tables[b])] = w.tables[b]
    lens = np.array(w.cached, dtype=np.int32)
    lens[7] = 10_000                       # beyond 16 * max_blocks: clamped and flagged
    out, ws = _attend(w.q.to(dev), w.k_cache.to(dev), w.v_cache.to(dev), torch.from_numpy(table).to(dev),
                      torch.from_numpy(lens).to(dev), w.scale)
    rc, flags = pkv.paged_decode_status(ws)
    assert rc == pkv.PKV_ERANGE and flags == 2
    lens[7] = 48
    ref = oracle.decode(w.q, "bf16", w.k_cache, w.v_cache, "bf16", table, np.maximum(lens, 0), scale=w.scale)
    compare(out, ref, "bf16", "large batch")


@pytest.mark.parametrize("dtype,q_dtype", [("bf16", "bf16"), ("f16", "f16"), ("fp8_e4m3", "bf16")])
def test_short_contexts_many_sequences(dtype, q_dtype):
    """Contexts of 1-8 tokens put single softmax weights near 1, where the
    rounding of the weights fed to the tensor cores would show directly."""
    spec = dict(B=1024, Hq=16, Hkv=2, D=128, dtype=dtype, q_dtype=q_dtype, ctx_range=(1, 8),
                free_frac=0.5, min_free=256)
    stats = _check_step(workloads.make(spec, seed=31))
    print(dtype, stats)


def test_sm_copy_between_pinned_host_and_device_is_exact():
    pkv = _pkv()
    g = torch.Generator().manual_seed(8)
    n = 3 * 1024 * 1024 + 48                    # not a multiple of the per-thread stride
    src_host = torch.randint(0, 256, (n,), generator=g, dtype=torch.uint8).pin_memory()
    dev = torch.empty(n, dtype=torch.uint8, device="cuda")
    back = torch.zeros(n, dtype=torch.uint8).pin_memory()
    pkv.pkv_copy(dev, src_host)                 # host -> device
    dev2 = torch.empty_like(dev)
    pkv.pkv_copy(dev2, dev)                     # device -> device
    pkv.pkv_copy(back, dev2)                    # device -> host
    torch.cuda.synchronize()
    assert torch.equal(back, src_host)
    with pytest.raises(pkv.PagedKVError):
        pkv.pkv_copy(dev, src_host, nbytes=7)   # not a multiple of 16 bytes


@pytest.mark.parametrize("spec", [
    dict(B=64, Hq=64, Hkv=8, D=128, dtype="bf16", ctx_range=(1, 3000)),                 # splits + merge
    dict(B=6, Hq=32, Hkv=32, D=128, dtype="f16", ctx_range=(1, 500)),                   # MHA (CUDA cores)
    dict(B=48, Hq=64, Hkv=8, D=128, dtype="bf16", q_len=4, ctx_range=(4, 9000)),        # tensor-core route
    dict(B=8, Hq=32, Hkv=8, D=128, dtype="fp8_e4m3", q_dtype="bf16", ctx_range=(1, 2000)),
], ids=lambda s: f"{s['dtype']}-q{s['Hq']}-kv{s['Hkv']}-L{s.get('q_len', 1)}")
def test_output_into_pinned_host_memory_is_identical(spec):
    """out may be pinned host memory: the kernels write the rows over the
    host link.  The bytes equal those of the same call into device memory."""
    pkv = _pkv()
    dev = "cuda"
    spec = dict(spec)
    spec.setdefault("q_dtype", spec["dtype"])
    spec.update(free_frac=0.2, min_free=4)
    w = workloads.make(spec, seed=83)
    table = np.full((w.B, w.max_blocks), -1, dtype=np.int32)
    for b in range(w.B):
        table[b, :len(w.tables[b])] = w.tables[b]
    args = (w.k_cache.to(dev), w.v_cache.to(dev), torch.from_numpy(table).to(dev),
            torch.tensor(w.context_lens, dtype=torch.int32, device=dev), w.scale,
            None if w.k_scale is None else w.k_scale.to(dev), None if w.v_scale is None else w.v_scale.to(dev))
    q = w.q.to(dev)
    d_out = torch.empty_like(q)
    h_out = torch.full(q.shape, float("nan"), dtype=q.dtype).pin_memory()
    pkv.paged_decode_attention(d_out, q, *args)
    pkv.paged_decode_attention(h_out, q, *args)
    torch.cuda.synchronize()
    assert torch.equal(d_out.cpu().view(torch.int16), h_out.view(torch.int16))
