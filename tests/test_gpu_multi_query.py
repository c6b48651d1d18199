"""GPU parity of multi-query paged decode: q_len new tokens per sequence
appended in one step and attended causally (new token i sees the cache up to
its own position — the verify step of speculative decoding, "LLM推理优化实战"
§4, with the mask tril(diagonal = kv_len - q_len) of "苦猿的大模型日记 Day45"
PART 04), through the C ABI against the oracle on the same seeded inputs."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_helpers import compare, routes, run_gpu_step, run_oracle_step

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
    assert np.array_equal(step.h_table.numpy(), table)
    assert np.array_equal(step.h_lens.numpy(), lens)
    assert np.array_equal(_bytes(step.k_cache).reshape(-1), kc.view(np.uint8).reshape(-1))
    assert np.array_equal(_bytes(step.v_cache).reshape(-1), vc.view(np.uint8).reshape(-1))
    if ks is not None:
        assert np.array_equal(step.k_scale.cpu().numpy(), ks)
        assert np.array_equal(step.v_scale.cpu().numpy(), vs)
    rc, flags = _pkv().paged_decode_status(step.workspace, step.stream)
    assert rc == 0 and flags == 0
    assert out.shape == ((w.B, w.q_len, w.Hq, w.D) if w.q.dim() == 4 else (w.B, w.Hq, w.D))
    return compare(out, ref, w.dtype, f"{w.name} q_len {w.q_len}")


@pytest.mark.parametrize("spec", [
    dict(Hq=16, Hkv=2, D=128, dtype="bf16", q_len=2, ctx=[40, 300, 2, 17]),
    dict(Hq=16, Hkv=2, D=128, dtype="bf16", q_len=4, ctx=[4, 16, 33, 700]),
    dict(Hq=16, Hkv=2, D=64, dtype="bf16", q_len=8, ctx=[8, 100, 250]),
    dict(Hq=8, Hkv=1, D=128, dtype="bf16", q_len=5, ctx=[5, 21, 160]),           # MQA, R = 40
    dict(Hq=6, Hkv=2, D=128, dtype="bf16", q_len=3, ctx=[3, 47, 129]),           # R = 9: 8 + 1
    dict(Hq=4, Hkv=4, D=128, dtype="f16", q_len=3, ctx=[3, 47, 129]),            # MHA, R = 3
    dict(Hq=8, Hkv=2, D=128, dtype="f16", q_len=6, ctx=[6, 90, 512]),
    dict(Hq=8, Hkv=2, D=128, dtype="fp8_e4m3", q_dtype="bf16", q_len=4, ctx=[19, 35, 4, 200]),
    dict(Hq=8, Hkv=2, D=64, dtype="fp8_e4m3", q_dtype="f16", q_len=2, ctx=[17, 2, 63]),
    dict(Hq=8, Hkv=2, D=128, dtype="f32", q_len=3, ctx=[3, 40, 177]),            # CUDA cores, GC 2
    dict(Hq=2, Hkv=2, D=64, dtype="f32", q_len=2, ctx=[2, 18, 33]),              # group 1, R = 2
], ids=lambda s: f"{s['dtype']}-q{s['Hq']}-kv{s['Hkv']}-d{s['D']}-L{s['q_len']}")
def test_multi_query_shapes_and_dtypes(spec):
    """Contexts cover ctx == q_len (nothing cached), tokens that open one or
    two blocks inside the step (fp8: a block's scale set by a token of the
    same call), ragged tails and several partition counts."""
    spec = dict(spec)
    spec.setdefault("q_dtype", spec["dtype"])
    spec["B"] = len(spec["ctx"])
    spec.update(free_frac=0.5, min_free=8)
    for seed, splits in ((5, 0), (6, 5), (7, 1000)):
        _check_step(workloads.make(spec, seed=seed), num_splits=splits)


@pytest.mark.parametrize("q_len", [2, 4, 8])
def test_multi_query_llama70b_layer(q_len):
    """The Llama-3.1-70B-shaped GQA-8 bf16 layer (Hq 64, Hkv 8, D 128) at
    context 8192 with q_len new tokens per sequence, 16 sequences, every
    output compared."""
    w = workloads.config(3, B=16, q_len=q_len)
    stats = _check_step(w)
    print(f"q_len {q_len}: {stats}")


def test_multi_query_full_size_workload():
    """64 sequences of 8192 positions (the bench's multi-query workload at
    q_len 4), every output compared."""
    stats = _check_step(workloads.config(3, q_len=4))
    print(stats)


def test_rows_that_see_nothing_are_zero():
    """A context shorter than q_len leaves the first rows of that sequence
    with no visible position: their output is 0, the others are exact."""
    pkv = _pkv()
    dev = "cuda"
    g = torch.Generator().manual_seed(12)
    B, L, Hq, Hkv, D, nb = 3, 4, 8, 2, 128, 6
    q = torch.randn((B, L, Hq, D), generator=g).to(torch.bfloat16)
    kc = torch.randn((nb, Hkv, 16, D), generator=g).to(torch.bfloat16)
    vc = torch.randn((nb, Hkv, 16, D), generator=g).to(torch.bfloat16)
    table = torch.tensor([[0, 1], [2, 3], [4, 5]], dtype=torch.int32)
    lens = torch.tensor([2, 0, 20], dtype=torch.int32)
    for splits in (0, 1, 7):
        out = torch.empty_like(q, device=dev)
        ws = pkv.paged_decode_attention(out, q.to(dev), kc.to(dev), vc.to(dev), table.to(dev),
                                        lens.to(dev), 0.1, num_splits=splits)
        rc, flags = pkv.paged_decode_status(ws)
        assert rc == 0 and flags == 0
        got = out.cpu()
        assert torch.all(got[0, :2] == 0) and torch.all(got[1] == 0)
        ref = oracle.decode(q, "bf16", kc, vc, "bf16", table.numpy(), lens.numpy(), scale=0.1)
        compare(out, ref, "bf16", f"short contexts, splits {splits}")


def test_q_len_one_in_4d_form_is_the_plain_decode():
    w = workloads.make(dict(B=5, Hq=16, Hkv=2, D=128, dtype="bf16", ctx_range=(1, 400),
                            free_frac=0.3), seed=41)
    pkv = _pkv()
    dev = "cuda"
    table = np.full((w.B, w.max_blocks), -1, dtype=np.int32)
    for b in range(w.B):
        table[b, :len(w.tables[b])] = w.tables[b]
    lens = torch.tensor(w.cached, dtype=torch.int32, device=dev)
    args = (w.k_cache.to(dev), w.v_cache.to(dev), torch.from_numpy(table).to(dev), lens, w.scale)
    q = w.q.to(dev)
    o3 = torch.empty_like(q)
    o4 = torch.empty_like(q)[:, None]
    pkv.paged_decode_attention(o3, q, *args)
    pkv.paged_decode_attention(o4, q[:, None].contiguous(), *args)
    torch.cuda.synchronize()
    assert torch.equal(o3, o4[:, 0])


def test_multi_token_append_into_shared_partial_block():
    """Two forks of a 390-token parent (24 full blocks + 6 tokens) append 3
    tokens each in one step: each copies the shared partial block once, then
    writes all three tokens into its copy; the parent is untouched
    ("LLM推理优化实战" §2.2 copy-on-write)."""
    from oracle.block_table import BlockTable
    from paged_kv_gqa_03_gb300.step import DecodeStep
    dev = "cuda"
    L, Hq, Hkv, D, nb = 3, 32, 8, 128, 40
    g = torch.Generator().manual_seed(19)
    kc = torch.randn((nb, Hkv, 16, D), generator=g).to(torch.bfloat16)
    vc = torch.randn((nb, Hkv, 16, D), generator=g).to(torch.bfloat16)
    q = torch.randn((2, L, Hq, D), generator=g).to(torch.bfloat16)
    kn = torch.randn((2, L, Hkv, D), generator=g).to(torch.bfloat16)
    vn = torch.randn((2, L, Hkv, D), generator=g).to(torch.bfloat16)
    step = DecodeStep(kc.to(dev), vc.to(dev), Hq, torch.bfloat16, 32, scale=0.09, q_len=L)
    ref_bt = BlockTable(nb)
    for bm in (step.bm, ref_bt):
        bm.allocate(0, 390)
        bm.fork(0, 1)
        bm.fork(0, 2)
    ncow = step.prepare([1, 2])
    step.upload()
    assert ncow == 2
    slots_ref, cow_ref = ref_bt.append_slots([1, 1, 1, 2, 2, 2])
    assert step.h_slots.tolist() == slots_ref
    assert [tuple(step.h_pairs[2 * i:2 * i + 2].tolist()) for i in range(2)] == cow_ref
    out = torch.empty((2, L, Hq, D), dtype=torch.bfloat16, device=dev)
    step.launch(q.to(dev), kn.to(dev), vn.to(dev), out)
    step.stream.synchronize()
    kr, vr = kc.clone(), vc.clone()
    for src, dst in cow_ref:
        kr[dst], vr[dst] = kr[src], vr[src]
    kr, vr, _, _ = oracle.append(kr, vr, "bf16", kn.reshape(-1, Hkv, D), vn.reshape(-1, Hkv, D),
                                 "bf16", slots_ref)
    assert np.array_equal(_bytes(step.k_cache), kr.view(np.uint8).reshape(_bytes(step.k_cache).shape))
    assert np.array_equal(_bytes(step.v_cache), vr.view(np.uint8).reshape(_bytes(step.v_cache).shape))
    table, lens = step.bm.export([1, 2], 32)
    assert lens.tolist() == [393, 393]
    ref = oracle.decode(q, "bf16", kr, vr, "bf16", table, lens, scale=0.09)
    compare(out, ref, "bf16", "multi-token cow")


def test_captured_multi_query_step_matches_eager():
    w = workloads.config(3, B=4, ctx=[700, 17, 33, 1500], free_frac=0.3, min_free=8, q_len=3)
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


@pytest.mark.parametrize("kernel", ["persistent", "tiles"])
@pytest.mark.parametrize("dtype,D,window", [("bf16", 128, 0), ("f16", 64, 0), ("bf16", 128, 37)])
def test_multi_query_tensor_core_route(dtype, D, window, kernel):
    """40 sequences x 4 kv heads (160 (sequence, kv head) tiles, one per SM or
    more): with num_splits = 0 the call takes a tensor-core prefill kernel
    (each of the two), with a fixed split count the 8-row-unit decode kernel;
    both against the oracle."""
    spec = dict(B=40, Hq=32, Hkv=4, D=D, dtype=dtype, q_len=5, ctx_range=(5, 300), free_frac=0.3,
                min_free=16, window=window)
    with routes(multi_query="prefill", prefill=kernel):
        for seed, splits in ((61, 0), (62, 7)):
            _check_step(workloads.make(spec, seed=seed), num_splits=splits)


@pytest.mark.parametrize("route", ["transposed", "prefill"])
@pytest.mark.parametrize("dtype,D,q_len,window", [("bf16", 128, 5, 0), ("bf16", 128, 3, 37), ("f16", 64, 4, 0)])
def test_multi_query_ragged_contexts_wide_table(dtype, D, q_len, window, route):
    """160 (sequence, kv head) items under a block table admitting 8000
    positions (one long sequence, so the one-CTA-per-item kernel with row
    replicas serves them) and ragged contexts (q_len .. 3000, many items of
    a single tile); every output against the oracle."""
    rng = np.random.default_rng(5)
    ctx = [8000] + [int(x) for x in rng.integers(q_len, 3000, 39)]
    spec = dict(B=40, Hq=32, Hkv=4, D=D, dtype=dtype, q_len=q_len, ctx=ctx, free_frac=0.2, min_free=16,
                window=window)
    with routes(multi_query="prefill" if route == "prefill" else "auto"):
        _check_step(workloads.make(spec, seed=71))


# The transposed tensor-core kernel (positions on the M side, stream-K over
# every (sequence, kv head) item's K / V tiles, the merge of items cut between
# CTAs) serves 16-bit caches with head dim 128: up to 32 query rows per kv head
# by default, up to 64 where the 128-row prefill route cannot fill the GPU.
@pytest.mark.parametrize("dtype,Hq,Hkv,q_len,ctx,window", [
    ("bf16", 2, 2, 2, [2, 130, 1000], 0),                   # MHA, R = 2 (16-row S^T, mostly padding)
    ("bf16", 16, 2, 2, [2, 129, 4000, 77], 0),              # R = 16
    ("f16", 16, 2, 2, [2, 129, 4000, 77], 0),
    ("bf16", 32, 4, 4, [4, 500, 2048, 3333, 7], 0),         # R = 32
    ("f16", 32, 4, 4, [4, 500, 2048, 3333, 7], 37),
    ("bf16", 40, 8, 7, [7, 300, 1500], 0),                  # R = 35: 64-row S^T
    ("bf16", 48, 3, 3, [3, 900, 260], 100),                 # R = 48, window
    ("bf16", 64, 8, 8, [8, 1200, 5000, 64], 0),             # R = 64
    ("f16", 64, 8, 8, [8, 1200, 5000, 64], 1),              # window 1: token i sees only itself
], ids=lambda v: str(v))
def test_transposed_kernel_rows_windows_dtypes(dtype, Hq, Hkv, q_len, ctx, window):
    """Every output against the oracle for 2 to 64 query rows per kv head
    (non-power-of-two counts padded), windows, bf16 (P as high part +
    residual) and f16; few items, so most CTAs' ranges are empty or cut an
    item."""
    spec = dict(B=len(ctx), Hq=Hq, Hkv=Hkv, D=128, dtype=dtype, q_len=q_len, ctx=ctx, free_frac=0.3,
                min_free=16, window=window)
    _check_step(workloads.make(spec, seed=81))


@pytest.mark.parametrize("ctx", [[100000], [60000, 4, 45000]])
def test_transposed_kernel_item_cut_across_every_cta(ctx):
    """One kv head of one long sequence holds most of the tiles, so its
    item is cut across (nearly) every CTA and the merge combines up to 152
    partials per row."""
    spec = dict(B=len(ctx), Hq=8, Hkv=1, D=128, dtype="bf16", q_len=4, ctx=ctx, free_frac=0.05, min_free=16)
    _check_step(workloads.make(spec, seed=83))


def test_transposed_kernel_flags_a_bad_block_id():
    """A block id past the pool reads as zeros and raises PKV_FLAG_BAD_BLOCK
    in the call's status; the other sequence is exact."""
    pkv = _pkv()
    dev = "cuda"
    g = torch.Generator().manual_seed(13)
    B, L, Hq, Hkv, D, nb = 2, 3, 8, 2, 128, 8
    q = torch.randn((B, L, Hq, D), generator=g).to(torch.bfloat16)
    kc = torch.randn((nb, Hkv, 16, D), generator=g).to(torch.bfloat16)
    vc = torch.randn((nb, Hkv, 16, D), generator=g).to(torch.bfloat16)
    table = torch.tensor([[0, 1, 2], [3, nb + 5, 4]], dtype=torch.int32)
    lens = torch.tensor([40, 40], dtype=torch.int32)
    out = torch.empty_like(q, device=dev)
    ws = pkv.paged_decode_attention(out, q.to(dev), kc.to(dev), vc.to(dev), table.to(dev), lens.to(dev), 0.1)
    rc, flags = pkv.paged_decode_status(ws)
    assert flags & pkv.PKV_FLAG_BAD_BLOCK
    ref = oracle.decode(q[:1], "bf16", kc, vc, "bf16", table[:1].numpy(), lens[:1].numpy(), scale=0.1)
    compare(out[:1], ref, "bf16", "the good sequence")


@pytest.mark.parametrize("q_len,B", [(4, 16), (8, 20)])
def test_transposed_kernel_equals_the_prefill_route(q_len, B):
    """The same 70B-shaped call (B sequences of 8192) through the transposed
    kernel and the 128-row prefill route, each forced: both within the bound
    of the oracle.  (At 64 rows with 160 items the prefill route is the
    default.)"""
    w = workloads.config(3, B=B, q_len=q_len)
    with routes(multi_query="transposed"):
        a = _check_step(w)
    with routes(multi_query="prefill"):
        b = _check_step(w)
    print(a, b)


# FP8 caches on the transposed kernel: each E4M3 tile is widened to f16 in
# shared memory by the producer warps (exact), the MMAs run on f16 (the query
# converted when staged), the block's K scale multiplies the scores and its V
# scale is folded into the weights; up to 32 query rows per kv head.
@pytest.mark.parametrize("q_dtype,Hq,Hkv,q_len,ctx,window", [
    ("bf16", 2, 2, 2, [2, 130, 1000], 0),                   # MHA, R = 2
    ("bf16", 16, 2, 2, [2, 129, 4000, 77], 0),              # R = 16
    ("f16", 16, 2, 2, [2, 129, 4000, 77], 0),
    ("bf16", 32, 4, 4, [4, 500, 2048, 3333, 7], 0),         # R = 32
    ("f16", 32, 4, 4, [4, 500, 2048, 3333, 7], 37),
    ("bf16", 24, 8, 7, [7, 300, 1500], 100),                # R = 21, window
    ("bf16", 32, 8, 8, [8, 1200, 5000, 64], 1),             # window 1: token i sees only itself
], ids=lambda v: str(v))
def test_transposed_kernel_fp8(q_dtype, Hq, Hkv, q_len, ctx, window):
    spec = dict(B=len(ctx), Hq=Hq, Hkv=Hkv, D=128, dtype="fp8_e4m3", q_dtype=q_dtype, q_len=q_len, ctx=ctx,
                free_frac=0.3, min_free=16, window=window)
    with routes(multi_query="transposed"):
        _check_step(workloads.make(spec, seed=91))


# FP8 caches with more than 8 query rows per kv head on the decode kernel:
# 16-row units (two 8-row column groups share each widened K / V fragment).
# Rows per unit 9-16 and a ragged second unit, D 64 and 128, bf16 and f16
# queries, windows, and fixed split counts (partials of 16-row units through
# the split-KV merge).
@pytest.mark.parametrize("q_dtype,Hq,Hkv,D,q_len,ctx,window", [
    ("bf16", 12, 3, 128, 3, [3, 47, 300, 1029], 0),          # R = 12: one unit, 4 rows unused
    ("f16", 8, 2, 64, 4, [4, 17, 64, 700], 0),               # R = 16, D 64
    ("bf16", 8, 1, 128, 3, [3, 200, 33], 0),                 # MQA, R = 24: units of 16 + 8 rows
    ("bf16", 32, 8, 128, 8, [8, 500, 2048, 77], 37),         # R = 32, window
    ("f16", 4, 2, 128, 5, [5, 99, 1000], 1),                 # R = 10, window 1
    ("bf16", 16, 1, 128, 1, [1, 40, 3000, 512], 0),          # q_len 1, group 16
    ("bf16", 12, 1, 64, 1, [7, 129, 2100], 100),             # q_len 1, group 12, window
], ids=lambda v: str(v))
def test_fp8_sixteen_row_units(q_dtype, Hq, Hkv, D, q_len, ctx, window):
    spec = dict(B=len(ctx), Hq=Hq, Hkv=Hkv, D=D, dtype="fp8_e4m3", q_dtype=q_dtype, q_len=q_len, ctx=ctx,
                free_frac=0.3, min_free=16, window=window)
    if q_len == 1:
        del spec["q_len"]  # the single-token form: q [B, Hq, D]
    with routes(multi_query="units"):
        for seed, splits in ((95, 0), (96, 5), (97, 1000)):
            _check_step(workloads.make(spec, seed=seed), num_splits=splits)


@pytest.mark.parametrize("route", ["transposed", "auto"])
def test_fp8_long_context_layer_multi_query(route):
    """The long-context fp8 layer (16 sequences of 32768 positions, Hq 32,
    Hkv 8) verifying 4 draft tokens per sequence (16 rows per kv head), on
    the transposed kernel (forced) and on the default route (the 16-row
    units); every output compared."""
    w = workloads.config(5, q_len=4)
    with routes(multi_query=route):
        print(_check_step(w))


def test_transposed_kernel_fp8_flags_a_bad_block_id():
    """A block id past the pool reads as zeros with scale 0 and raises
    PKV_FLAG_BAD_BLOCK; the other sequence is exact."""
    pkv = _pkv()
    dev = "cuda"
    w = workloads.make(dict(B=2, Hq=8, Hkv=2, D=128, dtype="fp8_e4m3", q_dtype="bf16", q_len=3, ctx=[40, 40],
                            free_frac=0.5, min_free=8), seed=93)
    table = np.full((2, 3), 0, dtype=np.int32)
    for b in range(2):
        table[b, :len(w.tables[b])] = w.tables[b]
    table[1, 1] = w.num_blocks + 5
    lens = np.array(w.cached, dtype=np.int32)
    q = w.q.to(dev)
    out = torch.empty_like(q)
    with routes(multi_query="transposed"):
        ws = pkv.paged_decode_attention(out, q, w.k_cache.to(dev), w.v_cache.to(dev), torch.from_numpy(table).to(dev),
                                        torch.from_numpy(lens).to(dev), w.scale, w.k_scale.to(dev), w.v_scale.to(dev))
    rc, flags = pkv.paged_decode_status(ws)
    assert flags & pkv.PKV_FLAG_BAD_BLOCK
    ref = oracle.decode(w.q[:1], "bf16", w.k_cache, w.v_cache, "fp8_e4m3", table[:1], lens[:1], scale=w.scale,
                        k_scale=w.k_scale.numpy(), v_scale=w.v_scale.numpy())
    compare(out[:1], ref, "fp8_e4m3", "the good sequence")


# Non-finite data where no attended position lies: every free pool block
# (the blocks a step's appends open) and every stale row past a context in
# its last block hold NaN, so a stale K row reaching a score unmasked, or a
# stale V row reaching P . V (0 * NaN), shows in the output.  The oracle
# reads attended positions only.
@pytest.mark.parametrize("dtype,q_dtype,Hq,Hkv,q_len,route", [
    ("bf16", "bf16", 64, 8, 1, "auto"),
    ("bf16", "bf16", 64, 8, 4, "auto"),          # transposed kernel
    ("bf16", "bf16", 16, 2, 4, "units"),         # 8-row units, q_len 4
    ("f16", "f16", 4, 4, 3, "auto"),
    ("fp8_e4m3", "bf16", 32, 8, 1, "auto"),      # 8-row fp8 units
    ("fp8_e4m3", "bf16", 32, 8, 4, "auto"),      # 16-row fp8 units
    ("fp8_e4m3", "f16", 16, 2, 5, "auto"),       # R = 40: 16 + 16 + 8 rows
    ("f32", "f32", 8, 2, 2, "auto"),             # CUDA cores
], ids=lambda v: str(v))
def test_stale_rows_and_free_blocks_hold_nan(dtype, q_dtype, Hq, Hkv, q_len, route):
    ctx = [q_len, 37, 300, 1000, 2051]
    spec = dict(B=len(ctx), Hq=Hq, Hkv=Hkv, D=128, dtype=dtype, q_dtype=q_dtype, ctx=ctx, free_frac=0.3,
                min_free=16)
    if q_len > 1:
        spec["q_len"] = q_len
    w = workloads.make(spec, seed=99)
    used = {blk for t in w.tables for blk in t}
    nan_byte = 0x7F  # E4M3 NaN
    for cache in (w.k_cache, w.v_cache):
        raw = cache.view(torch.uint8) if dtype == "fp8_e4m3" else None
        for blk in range(w.num_blocks):
            if blk not in used:
                if raw is not None:
                    raw[blk] = nan_byte
                else:
                    cache[blk] = float("nan")
        for b in range(w.B):
            end = w.cached[b] + w.q_len  # the context after this step's appends
            j, off = (end - 1) // 16, end % 16
            if off and j < len(w.tables[b]):
                if raw is not None:
                    raw[w.tables[b][j], :, off:] = nan_byte
                else:
                    cache[w.tables[b][j], :, off:] = float("nan")
    with routes(multi_query=route):
        _check_step(w)
