"""Pins of the oracle's attention against the pages' worked example, closed
forms, invariants and torch's scaled_dot_product_attention (a library routine
the oracle does not use)."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_inputs import dense_table, scatter, sdpa_reference

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _toy():
    with open(os.path.join(GOLDEN, "toy_attention_page4.json")) as f:
        return json.load(f)


def _f64(x):
    return torch.tensor(x, dtype=torch.float64)


def _oracle_f64(q, pool_k, pool_v, tables, max_blocks, ctx, block_size, scale, **kw):
    """Runs the oracle on float64 inputs stored as f32 (tests choose values that
    are exact in f32 or compare against f32-rounded references)."""
    return oracle.decode(q.float().numpy(), "f32", pool_k.float().numpy(), pool_v.float().numpy(),
                         "f32", dense_table(tables, max_blocks), ctx, scale=scale,
                         block_size=block_size, **kw)


@pytest.mark.parametrize("block_size", [1, 2, 16])
def test_toy_incremental_step_equals_full_recompute(block_size):
    """Page 'KV Cache篇' §2.1/§2.2: predicting '好' from '天气真' with cached K/V
    of '天气' plus the new row gives the newest row of the full masked
    computation; the first two rows of step 2 are the rows of step 1."""
    t = _toy()
    X1, X2 = _f64(t["X_step1"]), _f64(t["X_step2"])
    WQ, WK, WV = _f64(t["W_Q"]), _f64(t["W_K"]), _f64(t["W_V"])
    div = t["scale_divisor"]
    # the page's own steps (Q = X @ W_Q, no transpose), rounded to f32 storage
    Q2, K2, V2 = [(X2 @ W).float().double() for W in (WQ, WK, WV)]
    mask = torch.triu(torch.full((3, 3), float("-inf"), dtype=torch.float64), diagonal=1)
    full = torch.softmax(Q2 @ K2.T / div + mask, dim=-1) @ V2           # the page's formulation
    sdpa = torch.nn.functional.scaled_dot_product_attention(
        Q2[None], K2[None], V2[None], is_causal=True, scale=1.0 / div)[0]
    assert torch.allclose(full, sdpa, rtol=0, atol=1e-14)
    # step 1 on its own gives the first two rows
    Q1, K1, V1 = [(X1 @ W).float().double() for W in (WQ, WK, WV)]
    mask1 = torch.triu(torch.full((2, 2), float("-inf"), dtype=torch.float64), diagonal=1)
    step1 = torch.softmax(Q1 @ K1.T / div + mask1, dim=-1) @ V1
    assert torch.allclose(step1, full[:2], rtol=0, atol=1e-15)

    # incremental decode: cache rows 0..1 (step 1), append row 2, attend row 2
    Hkv, D = 1, 4
    n3 = (3 + block_size - 1) // block_size
    nblk = n3 + 1
    perm = np.random.default_rng(5).permutation(nblk)
    pool_k, tables, mb = scatter([K2[:2, None, :]], Hkv, D, block_size, nblk, perm)
    pool_v, _, _ = scatter([V2[:2, None, :]], Hkv, D, block_size, nblk, perm)
    # the table once it has room for the third token, and that token's slot
    t2 = [int(perm[i]) for i in range(n3)]
    assert t2[:len(tables[0])] == tables[0]
    slot = t2[2 // block_size] * block_size + 2 % block_size
    kc, vc, _, _ = oracle.append(pool_k.float().numpy(), pool_v.float().numpy(), "f32",
                                 K2[2:3, None, :].float().numpy(), V2[2:3, None, :].float().numpy(),
                                 "f32", [slot], block_size=block_size)
    bt = dense_table([t2], len(t2))
    q = Q2[2:3, None, :].float().numpy()
    out = oracle.decode(q, "f32", kc, vc, "f32", bt, [3], scale=1.0 / div, block_size=block_size)
    assert np.allclose(out[0, 0], full[2].numpy(), rtol=0, atol=1e-12)
    # the second row: query 1 over the first two cached positions
    out2 = oracle.decode(Q2[1:2, None, :].float().numpy(), "f32", kc, vc, "f32", bt, [2],
                         scale=1.0 / div, block_size=block_size)
    assert np.allclose(out2[0, 0], full[1].numpy(), rtol=0, atol=1e-12)
    # first row: one visible key, so the output is V row 0 exactly
    out1 = oracle.decode(Q2[0:1, None, :].float().numpy(), "f32", kc, vc, "f32", bt, [1],
                         scale=1.0 / div, block_size=block_size)
    assert np.array_equal(out1[0, 0], V2[0].numpy())


def _random_case(seed, B, Hq, Hkv, D, block_size, max_ctx, spare=3):
    g = torch.Generator().manual_seed(seed)
    ctx = torch.randint(1, max_ctx + 1, (B,), generator=g).tolist()
    ks = [torch.randn((c, Hkv, D), generator=g, dtype=torch.float64).float().double() for c in ctx]
    vs = [torch.randn((c, Hkv, D), generator=g, dtype=torch.float64).float().double() for c in ctx]
    q = torch.randn((B, Hq, D), generator=g, dtype=torch.float64).float().double()
    nb = sum((c + block_size - 1) // block_size for c in ctx) + spare
    perm = torch.randperm(nb, generator=g).numpy()
    return ctx, ks, vs, q, nb, perm


@pytest.mark.parametrize("B,Hq,Hkv,D,bs,max_ctx", [
    (3, 4, 2, 8, 16, 40),      # GQA group 2
    (2, 8, 1, 16, 4, 37),      # MQA
    (4, 3, 3, 8, 2, 19),       # MHA (group 1)
    (2, 16, 2, 64, 16, 70),    # group 8
])
def test_bruteforce_matches_sdpa(B, Hq, Hkv, D, bs, max_ctx):
    ctx, ks, vs, q, nb, perm = _random_case(11 + B * Hq, B, Hq, Hkv, D, bs, max_ctx)
    pk, tables, mb = scatter(ks, Hkv, D, bs, nb, perm)
    pv, _, _ = scatter(vs, Hkv, D, bs, nb, perm)
    scale = 1.0 / math.sqrt(D)
    got = _oracle_f64(q, pk, pv, tables, mb, ctx, bs, scale)
    ref = sdpa_reference(q, ks, vs, scale).numpy()
    assert np.allclose(got, ref, rtol=0, atol=1e-12)


def test_closed_forms():
    D, Hkv, Hq, bs = 8, 1, 2, 4
    g = torch.Generator().manual_seed(3)
    q = torch.randn((1, Hq, D), generator=g, dtype=torch.float64).float().double()
    V = torch.randn((11, Hkv, D), generator=g, dtype=torch.float64).float().double()
    perm = np.arange(3)
    pv, tables, mb = scatter([V], Hkv, D, bs, 3, perm)
    # all keys equal -> uniform weights -> mean of V
    Keq = torch.ones((11, Hkv, D), dtype=torch.float64)
    pk, _, _ = scatter([Keq], Hkv, D, bs, 3, perm)
    out = _oracle_f64(q, pk, pv, tables, mb, [11], bs, 0.5)
    assert np.allclose(out[0, 0], V[:, 0].mean(0).numpy(), atol=1e-14)
    # one key aligned with q far above the rest -> output is that key's value
    K = torch.zeros((11, Hkv, D), dtype=torch.float64)
    K[7, 0] = 50.0 * q[0, 0]
    pk, _, _ = scatter([K], Hkv, D, bs, 3, perm)
    out = _oracle_f64(q, pk, pv, tables, mb, [11], bs, 1.0)
    assert np.allclose(out[0, 0], V[7, 0].numpy(), atol=1e-12)
    # context of one -> output equals V_0 for every head
    out = _oracle_f64(q, pk, pv, tables, mb, [1], bs, 1.0)
    assert np.array_equal(out[0, 0], V[0, 0].numpy()) and np.array_equal(out[0, 1], V[0, 0].numpy())
    # context of zero -> zeros and lse = -inf
    out, lse = _oracle_f64(q, pk, pv, tables, mb, [0], bs, 1.0, with_lse=True)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_scores_scale_and_head_mapping():
    """Two keys with scores s and 0 give weight sigmoid(s) on the first; heads
    1..G-1 of a group must read kv head 0 and heads G.. kv head 1."""
    D, bs = 4, 16
    K = torch.zeros((2, 2, D), dtype=torch.float64)
    V = torch.zeros((2, 2, D), dtype=torch.float64)
    K[0, 0, 0], K[0, 1, 1] = 1.0, 1.0
    V[0, :, 2], V[1, :, 3] = 1.0, 1.0
    V[0, 1, 2] = 2.0                      # kv head 1 has a different value row
    q = torch.zeros((1, 4, D), dtype=torch.float64)
    q[0, 0, 0], q[0, 1, 0], q[0, 2, 1], q[0, 3, 0] = 3.0, 1.0, 2.0, 5.0
    pk, tables, mb = scatter([K], 2, D, bs, 1, [0])
    pv, _, _ = scatter([V], 2, D, bs, 1, [0])
    scale = 0.5
    out = _oracle_f64(q, pk, pv, tables, mb, [2], bs, scale)
    sig = lambda s: 1.0 / (1.0 + math.exp(-s))
    assert math.isclose(out[0, 0, 2], sig(3.0 * scale), abs_tol=1e-14)   # head 0 -> kv 0
    assert math.isclose(out[0, 1, 2], sig(1.0 * scale), abs_tol=1e-14)   # head 1 -> kv 0
    assert math.isclose(out[0, 2, 2], 2.0 * sig(2.0 * scale), abs_tol=1e-14)  # head 2 -> kv 1
    assert math.isclose(out[0, 3, 2], 2.0 * sig(0.0), abs_tol=1e-14)     # head 3 -> kv 1: q.k = 0
    assert math.isclose(out[0, 3, 3], 1.0 - sig(0.0), abs_tol=1e-14)


def test_block_permutation_invariance():
    B, Hq, Hkv, D, bs = 3, 4, 2, 8, 16
    ctx, ks, vs, q, nb, perm = _random_case(21, B, Hq, Hkv, D, bs, 70)
    scale = 0.3
    outs = []
    for p in (perm, perm[::-1].copy(), np.random.default_rng(1).permutation(nb)):
        pk, tables, mb = scatter(ks, Hkv, D, bs, nb, p)
        pv, _, _ = scatter(vs, Hkv, D, bs, nb, p)
        outs.append(_oracle_f64(q, pk, pv, tables, mb, ctx, bs, scale))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_shared_prefix_equals_copied_prefix():
    """Sequences whose tables reference the same prefix blocks give the same
    result as sequences holding private copies ('LLM推理优化实战' §2.2 CoW)."""
    Hq, Hkv, D, bs = 4, 2, 8, 4
    g = torch.Generator().manual_seed(4)
    pre_k = torch.randn((8, Hkv, D), generator=g, dtype=torch.float64).float().double()
    pre_v = torch.randn((8, Hkv, D), generator=g, dtype=torch.float64).float().double()
    suf = [5, 9, 2]
    ks = [torch.cat([pre_k, torch.randn((s, Hkv, D), generator=g).double()]) for s in suf]
    vs = [torch.cat([pre_v, torch.randn((s, Hkv, D), generator=g).double()]) for s in suf]
    q = torch.randn((3, Hq, D), generator=g, dtype=torch.float64).float().double()
    ctx = [8 + s for s in suf]
    # copied: every sequence has its own prefix blocks
    nb = sum((c + bs - 1) // bs for c in ctx)
    pk, tables, mb = scatter(ks, Hkv, D, bs, nb, np.arange(nb))
    pv, _, _ = scatter(vs, Hkv, D, bs, nb, np.arange(nb))
    copied = _oracle_f64(q, pk, pv, tables, mb, ctx, bs, 0.4)
    # shared: the two prefix blocks of sequence 0 are referenced by all three
    shared_tables = [tables[0]] + [tables[0][:2] + t[2:] for t in tables[1:]]
    pk[tables[1][0]] = 0; pk[tables[1][1]] = 0; pk[tables[2][0]] = 0; pk[tables[2][1]] = 0
    shared = _oracle_f64(q, pk, pv, shared_tables, mb, ctx, bs, 0.4)
    assert np.array_equal(copied, shared)


def test_merge_of_partials_equals_full():
    B, Hq, Hkv, D, bs = 2, 4, 2, 8, 4
    ctx, ks, vs, q, nb, perm = _random_case(31, B, Hq, Hkv, D, bs, 45)
    ctx = [max(c, 9) for c in ctx]
    ks = [torch.cat([k, torch.randn((9, Hkv, D), dtype=torch.float64)])[:c] for k, c in zip(ks, ctx)]
    vs = [torch.cat([v, torch.randn((9, Hkv, D), dtype=torch.float64)])[:c] for v, c in zip(vs, ctx)]
    nb = sum((c + bs - 1) // bs for c in ctx) + 2
    perm = np.random.default_rng(2).permutation(nb)
    pk, tables, mb = scatter(ks, Hkv, D, bs, nb, perm)
    pv, _, _ = scatter(vs, Hkv, D, bs, nb, perm)
    scale = 0.35
    full = _oracle_f64(q, pk, pv, tables, mb, ctx, bs, scale)
    rng = np.random.default_rng(8)
    for S in (1, 2, 3, 5):
        cuts = [sorted(rng.choice(np.arange(1, c), S - 1, replace=False).tolist()) if S > 1 else []
                for c in ctx]
        o_parts = np.zeros((B, Hq, S + 1, D))
        lse_parts = np.full((B, Hq, S + 1), -np.inf)   # one extra empty partial
        for s in range(S):
            t0 = [([0] + c)[s] for c in cuts]
            t1 = [(c + [n])[s] for c, n in zip(cuts, ctx)]
            o, l = _oracle_f64(q, pk, pv, tables, mb, t1, bs, scale, t_begin=t0, with_lse=True)
            o_parts[:, :, s], lse_parts[:, :, s] = o, l
        merged = oracle.merge(o_parts.reshape(B * Hq, S + 1, D), lse_parts.reshape(B * Hq, S + 1))
        assert np.allclose(merged.reshape(B, Hq, D), full, rtol=0, atol=1e-13)
    # an all-empty row merges to zeros
    assert np.all(oracle.merge(np.ones((1, 2, D)), np.full((1, 2), -np.inf)) == 0)


def test_fp8_cache_is_dequantised_bytes_times_scale():
    """An fp8 cache attends over decode(byte) * scale[block, head]; compared
    with SDPA on those values computed by torch's float8 conversion."""
    g = torch.Generator().manual_seed(12)
    B, Hq, Hkv, D, bs, nb = 2, 4, 2, 16, 16, 5
    codes = torch.randint(0, 256, (nb, Hkv, bs, D), generator=g, dtype=torch.uint8)
    codes[(codes & 0x7f) == 0x7f] = 0x3c          # no NaN codes
    ksc = torch.rand((nb, Hkv), generator=g) + 0.01
    vsc = torch.rand((nb, Hkv), generator=g) + 0.01
    vcodes = codes.flip(-1).contiguous()
    tables = [[3, 0], [4, 1, 2]]
    ctx = [20, 41]
    q = torch.randn((B, Hq, D), generator=g).to(torch.bfloat16)
    got = oracle.decode(q, "bf16", codes.numpy(), vcodes.numpy(), "fp8_e4m3",
                        dense_table(tables, 3), ctx, scale=0.25,
                        k_scale=ksc.numpy(), v_scale=vsc.numpy())
    kd = codes.view(torch.float8_e4m3fn).double() * ksc.double()[:, :, None, None]
    vd = vcodes.view(torch.float8_e4m3fn).double() * vsc.double()[:, :, None, None]
    ks = [torch.stack([kd[tables[b][t // bs], :, t % bs] for t in range(ctx[b])]) for b in range(B)]
    vs = [torch.stack([vd[tables[b][t // bs], :, t % bs] for t in range(ctx[b])]) for b in range(B)]
    ref = sdpa_reference(q.double(), ks, vs, 0.25).numpy()
    assert np.allclose(got, ref, rtol=0, atol=1e-12)


def _multi_case(seed, B, q_len, Hq, Hkv, D, bs, max_ctx):
    g = torch.Generator().manual_seed(seed)
    ctx = torch.randint(q_len, max_ctx + 1, (B,), generator=g).tolist()
    ks = [torch.randn((c, Hkv, D), generator=g, dtype=torch.float64).float().double() for c in ctx]
    vs = [torch.randn((c, Hkv, D), generator=g, dtype=torch.float64).float().double() for c in ctx]
    q = torch.randn((B, q_len, Hq, D), generator=g, dtype=torch.float64).float().double()
    nb = sum((c + bs - 1) // bs for c in ctx) + 2
    perm = torch.randperm(nb, generator=g).numpy()
    pk, tables, mb = scatter(ks, Hkv, D, bs, nb, perm)
    pv, _, _ = scatter(vs, Hkv, D, bs, nb, perm)
    return ctx, ks, vs, q, pk, pv, tables, mb


@pytest.mark.parametrize("B,q_len,Hq,Hkv,D,bs,max_ctx", [
    (3, 2, 8, 2, 16, 16, 40),
    (2, 4, 8, 1, 8, 4, 37),      # MQA, small blocks
    (2, 5, 16, 2, 64, 16, 70),   # group 8
    (2, 3, 3, 3, 8, 2, 9),       # MHA, contexts down to q_len
])
def test_multi_query_matches_masked_sdpa(B, q_len, Hq, Hkv, D, bs, max_ctx):
    """q_len new tokens per sequence (the verify step of speculative decoding,
    'LLM推理优化实战' §4): new token i sees the cache up to its own position, the
    mask tril(ones(q_len, kv_len), diagonal = kv_len - q_len) of the
    naive_attention of '苦猿的大模型日记 Day45' PART 04, given to torch SDPA as a
    boolean mask."""
    ctx, ks, vs, q, pk, pv, tables, mb = _multi_case(7 + q_len * B, B, q_len, Hq, Hkv, D, bs,
                                                     max_ctx)
    scale = 1.0 / math.sqrt(D)
    got, lse = oracle.decode(q.float().numpy(), "f32", pk.float().numpy(), pv.float().numpy(),
                             "f32", dense_table(tables, mb), ctx, scale=scale, block_size=bs,
                             with_lse=True)
    assert got.shape == (B, q_len, Hq, D) and lse.shape == (B, q_len, Hq)
    G = Hq // Hkv
    for b in range(B):
        T = ctx[b]
        mask = torch.tril(torch.ones((q_len, T), dtype=torch.bool), diagonal=T - q_len)
        Kx = ks[b].permute(1, 0, 2).repeat_interleave(G, dim=0)      # [Hq, T, D]
        Vx = vs[b].permute(1, 0, 2).repeat_interleave(G, dim=0)
        Qx = q[b].permute(1, 0, 2)                                     # [Hq, q_len, D]
        ref = torch.nn.functional.scaled_dot_product_attention(Qx, Kx, Vx, attn_mask=mask,
                                                               scale=scale)
        assert np.allclose(got[b], ref.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)
        s = (Qx @ Kx.transpose(1, 2)) * scale
        ref_lse = torch.logsumexp(s.masked_fill(~mask, float("-inf")), dim=-1)   # [Hq, q_len]
        assert np.allclose(lse[b], ref_lse.T.numpy(), rtol=0, atol=1e-12)


def test_multi_query_rows_are_single_queries_over_shorter_contexts():
    """Token i of q_len equals a one-query decode whose context stops at its
    own position; q_len = 1 in the 4-D form equals the 3-D form bit for bit."""
    B, q_len, Hq, Hkv, D, bs = 3, 4, 4, 2, 8, 4
    ctx, ks, vs, q, pk, pv, tables, mb = _multi_case(19, B, q_len, Hq, Hkv, D, bs, 30)
    bt = dense_table(tables, mb)
    args = (pk.float().numpy(), pv.float().numpy(), "f32", bt)
    multi = oracle.decode(q.float().numpy(), "f32", *args, ctx, scale=0.3, block_size=bs)
    for i in range(q_len):
        one = oracle.decode(q[:, i].float().numpy(), "f32", *args,
                            [c - (q_len - 1 - i) for c in ctx], scale=0.3, block_size=bs)
        assert np.array_equal(multi[:, i], one)
    single = oracle.decode(q[:, :1].float().numpy(), "f32", *args, ctx, scale=0.3, block_size=bs)
    plain = oracle.decode(q[:, 0].float().numpy(), "f32", *args, ctx, scale=0.3, block_size=bs)
    assert np.array_equal(single[:, 0], plain)


def test_multi_query_toy_rows_of_full_masked_computation():
    """Page 'KV Cache篇' §2.1: with '天' cached and '气真' both new, the two new
    rows are rows 1 and 2 of the full causally masked computation."""
    t = _toy()
    X2 = _f64(t["X_step2"])
    WQ, WK, WV = _f64(t["W_Q"]), _f64(t["W_K"]), _f64(t["W_V"])
    div = t["scale_divisor"]
    Q2, K2, V2 = [(X2 @ W).float().double() for W in (WQ, WK, WV)]
    mask = torch.triu(torch.full((3, 3), float("-inf"), dtype=torch.float64), diagonal=1)
    full = torch.softmax(Q2 @ K2.T / div + mask, dim=-1) @ V2
    pk, tables, mb = scatter([K2[:, None, :]], 1, 4, 2, 2, [1, 0])
    pv, _, _ = scatter([V2[:, None, :]], 1, 4, 2, 2, [1, 0])
    q = Q2[1:3][None, :, None, :]                                         # [1, 2, 1, 4]
    out = oracle.decode(q.float().numpy(), "f32", pk.float().numpy(), pv.float().numpy(), "f32",
                        dense_table(tables, mb), [3], scale=1.0 / div, block_size=2)
    assert np.allclose(out[0, :, 0], full[1:3].numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("B,q_len,window,Hq,Hkv,D,bs,max_ctx", [
    (3, 1, 5, 8, 2, 16, 16, 60),
    (3, 1, 17, 4, 2, 8, 4, 70),
    (2, 4, 6, 8, 1, 8, 4, 37),       # several new tokens, each with its own window
    (2, 3, 16, 16, 2, 64, 16, 90),
])
def test_sliding_window_matches_band_masked_sdpa(B, q_len, window, Hq, Hkv, D, bs, max_ctx):
    """Sliding window ('苦猿的大模型日记 Day45' PART 02, third advanced
    direction): a row sees the `window` most recent positions up to its own,
    i.e. the causal mask of PART 04 intersected with triu(diagonal =
    kv_len - q_len - window + 1); compared with torch SDPA on that mask."""
    ctx, ks, vs, q, pk, pv, tables, mb = _multi_case(3 + window + q_len, B, q_len, Hq, Hkv, D, bs,
                                                     max_ctx)
    scale = 1.0 / math.sqrt(D)
    got, lse = oracle.decode(q.float().numpy(), "f32", pk.float().numpy(), pv.float().numpy(),
                             "f32", dense_table(tables, mb), ctx, scale=scale, block_size=bs,
                             with_lse=True, window=window)
    G = Hq // Hkv
    for b in range(B):
        T = ctx[b]
        causal = torch.tril(torch.ones((q_len, T), dtype=torch.bool), diagonal=T - q_len)
        band = torch.triu(torch.ones((q_len, T), dtype=torch.bool), diagonal=T - q_len - window + 1)
        mask = causal & band
        Kx = ks[b].permute(1, 0, 2).repeat_interleave(G, dim=0)
        Vx = vs[b].permute(1, 0, 2).repeat_interleave(G, dim=0)
        Qx = q[b].permute(1, 0, 2)
        ref = torch.nn.functional.scaled_dot_product_attention(Qx, Kx, Vx, attn_mask=mask,
                                                               scale=scale)
        assert np.allclose(got[b], ref.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)
        s = (Qx @ Kx.transpose(1, 2)) * scale
        ref_lse = torch.logsumexp(s.masked_fill(~mask, float("-inf")), dim=-1)
        assert np.allclose(lse[b], ref_lse.T.numpy(), rtol=0, atol=1e-12)


def test_sliding_window_special_cases():
    """A window covering the context is no window (bit for bit); a window of
    one gives each row its own position's V exactly; blocks wholly before
    every row's window are never read (their table entries may be -1)."""
    B, q_len, Hq, Hkv, D, bs = 3, 2, 4, 2, 8, 4
    ctx, ks, vs, q, pk, pv, tables, mb = _multi_case(29, B, q_len, Hq, Hkv, D, bs, 45)
    bt = dense_table(tables, mb)
    args = (pk.float().numpy(), pv.float().numpy(), "f32")
    qf = q.float().numpy()
    full = oracle.decode(qf, "f32", *args, bt, ctx, scale=0.3, block_size=bs)
    wide = oracle.decode(qf, "f32", *args, bt, ctx, scale=0.3, block_size=bs, window=max(ctx))
    assert np.array_equal(full, wide)
    one = oracle.decode(qf, "f32", *args, bt, ctx, scale=0.3, block_size=bs, window=1)
    for b in range(B):
        for i in range(q_len):
            pos = ctx[b] - q_len + i
            for hq in range(Hq):
                assert np.array_equal(one[b, i, hq], vs[b][pos, hq // (Hq // Hkv)].numpy())
    W = 5
    ref = oracle.decode(qf, "f32", *args, bt, ctx, scale=0.3, block_size=bs, window=W)
    holed = bt.copy()
    for b in range(B):
        first = max(0, ctx[b] - (q_len - 1) - W)       # earliest position any row sees
        holed[b, :first // bs] = -1
    got = oracle.decode(qf, "f32", *args, holed, ctx, scale=0.3, block_size=bs, window=W)
    assert np.array_equal(got, ref)


def test_prefill_matches_causal_sdpa_over_the_prompt():
    """Prefill with nothing cached: each sequence's whole prompt attends
    causally to itself — torch SDPA with is_causal on the contiguous K/V
    ('LLM推理优化实战' §3.2 flash_attention computes exactly this), with GQA."""
    g = torch.Generator().manual_seed(41)
    Hq, Hkv, D, bs = 8, 2, 16, 4
    n = [1, 7, 16, 23]
    ks = [torch.randn((t, Hkv, D), generator=g, dtype=torch.float64).float().double() for t in n]
    vs = [torch.randn((t, Hkv, D), generator=g, dtype=torch.float64).float().double() for t in n]
    q = torch.randn((sum(n), Hq, D), generator=g, dtype=torch.float64).float().double()
    nb = sum((t + bs - 1) // bs for t in n) + 1
    perm = torch.randperm(nb, generator=g).numpy()
    pk, tables, mb = scatter(ks, Hkv, D, bs, nb, perm)
    pv, _, _ = scatter(vs, Hkv, D, bs, nb, perm)
    q_start = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    got = oracle.prefill(q.float().numpy(), "f32", pk.float().numpy(), pv.float().numpy(), "f32",
                         dense_table(tables, mb), n, q_start, scale=0.25, block_size=bs)
    G = Hq // Hkv
    for b in range(len(n)):
        Qx = q[q_start[b]:q_start[b + 1]].permute(1, 0, 2)
        Kx = ks[b].permute(1, 0, 2).repeat_interleave(G, dim=0)
        Vx = vs[b].permute(1, 0, 2).repeat_interleave(G, dim=0)
        ref = torch.nn.functional.scaled_dot_product_attention(Qx, Kx, Vx, is_causal=True, scale=0.25)
        assert np.allclose(got[q_start[b]:q_start[b + 1]], ref.permute(1, 0, 2).numpy(), rtol=0,
                           atol=1e-12)


def test_prefill_with_cached_prefix_equals_multi_query_rows():
    """A prompt chunk after a cached prefix (chunked prefill): with every n_b
    equal to L the packed prefill equals the multi-query decode bit for bit;
    ragged n_b equal per-sequence multi-query calls, windows included."""
    B, L, Hq, Hkv, D, bs = 3, 5, 4, 2, 8, 4
    ctx, ks, vs, q, pk, pv, tables, mb = _multi_case(53, B, L, Hq, Hkv, D, bs, 60)
    bt = dense_table(tables, mb)
    args = (pk.float().numpy(), pv.float().numpy(), "f32", bt, ctx)
    for W in (0, 7):
        multi = oracle.decode(q.float().numpy(), "f32", *args, scale=0.3, block_size=bs, window=W)
        packed = oracle.prefill(q.reshape(B * L, Hq, D).float().numpy(), "f32", *args,
                                np.arange(0, B * L + 1, L), scale=0.3, block_size=bs, window=W)
        assert np.array_equal(packed.reshape(B, L, Hq, D), multi)
    n = [2, 5, 1]
    q_start = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    rows = torch.cat([q[b, L - n[b]:] for b in range(B)])       # the last n_b new tokens
    got = oracle.prefill(rows.float().numpy(), "f32", *args, q_start, scale=0.3, block_size=bs)
    for b in range(B):
        one = oracle.decode(q[b:b + 1, L - n[b]:].float().numpy(), "f32", pk.float().numpy(),
                            pv.float().numpy(), "f32", bt[b:b + 1], ctx[b:b + 1], scale=0.3,
                            block_size=bs)
        assert np.array_equal(got[q_start[b]:q_start[b + 1]], one[0])


def test_prefill_toy_example_is_the_full_masked_computation():
    """Page 'KV Cache篇' §2.1: prefilling all three tokens of '天气真' gives the
    page's full causally masked computation, row for row."""
    t = _toy()
    X2 = _f64(t["X_step2"])
    WQ, WK, WV = _f64(t["W_Q"]), _f64(t["W_K"]), _f64(t["W_V"])
    div = t["scale_divisor"]
    Q2, K2, V2 = [(X2 @ W).float().double() for W in (WQ, WK, WV)]
    mask = torch.triu(torch.full((3, 3), float("-inf"), dtype=torch.float64), diagonal=1)
    full = torch.softmax(Q2 @ K2.T / div + mask, dim=-1) @ V2
    pk, tables, mb = scatter([K2[:, None, :]], 1, 4, 2, 2, [1, 0])
    pv, _, _ = scatter([V2[:, None, :]], 1, 4, 2, 2, [1, 0])
    out = oracle.prefill(Q2[:, None, :].float().numpy(), "f32", pk.float().numpy(),
                         pv.float().numpy(), "f32", dense_table(tables, mb), [3], [0, 3],
                         scale=1.0 / div, block_size=2)
    assert np.allclose(out[:, 0], full.numpy(), rtol=0, atol=1e-12)
