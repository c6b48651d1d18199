"""Pins of the oracle's append step, the KV-bytes formula (the pages' worked
numbers) and the pure-Python block table (the page's BlockTable semantics)."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from oracle.block_table import BlockTable

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_append_writes_exactly_the_slots(dtype):
    tt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dtype]
    g = torch.Generator().manual_seed(1)
    nb, Hkv, D, B = 6, 2, 8, 3
    kc = torch.randn((nb, Hkv, 16, D), generator=g).to(tt)
    vc = torch.randn((nb, Hkv, 16, D), generator=g).to(tt)
    kn = torch.randn((B, Hkv, D), generator=g).to(tt)
    vn = torch.randn((B, Hkv, D), generator=g).to(tt)
    slots = [5 * 16 + 3, -1, 2 * 16 + 15]
    k2, v2, _, _ = oracle.append(kc, vc, dtype, kn, vn, dtype, slots)
    view = (lambda t: t.view(torch.int16).numpy()) if dtype != "f32" else (lambda t: t.numpy())
    k_ref, v_ref = view(kc).copy(), view(vc).copy()
    for b, s in enumerate(slots):
        if s >= 0:
            k_ref[s // 16, :, s % 16] = view(kn)[b]
            v_ref[s // 16, :, s % 16] = view(vn)[b]
    assert np.array_equal(k2.view(k_ref.dtype), k_ref)
    assert np.array_equal(v2.view(v_ref.dtype), v_ref)


def test_append_fp8_uses_block_scale_or_opens_block():
    g = torch.Generator().manual_seed(2)
    nb, Hkv, D = 4, 2, 16
    kc = torch.randint(0, 0x7e, (nb, Hkv, 16, D), generator=g, dtype=torch.uint8)
    vc = kc.clone()
    ks = torch.rand((nb, Hkv), generator=g) * 0.02 + 0.001
    vs = torch.rand((nb, Hkv), generator=g) * 0.02 + 0.001
    kn = (torch.randn((2, Hkv, D), generator=g) * 3).to(torch.bfloat16)
    vn = (torch.randn((2, Hkv, D), generator=g) * 3).to(torch.bfloat16)
    slots = [1 * 16 + 7, 3 * 16 + 0]          # existing block; block-opening token
    k2, v2, ks2, vs2 = oracle.append(kc.numpy(), vc.numpy(), "fp8_e4m3", kn, vn, "bf16",
                                     slots, k_scale=ks.numpy(), v_scale=vs.numpy())
    for src, cache, sc_in, sc_out in ((kn, k2, ks, ks2), (vn, v2, vs, vs2)):
        x = src.float()
        # existing block: fp32 division by the stored scale, torch's RNE cast
        r = (x[0] / sc_in[1][:, None]).clamp(-448, 448)
        assert np.array_equal(cache[1, :, 7], r.to(torch.float8_e4m3fn).view(torch.uint8).numpy())
        assert np.array_equal(sc_out[1], sc_in[1].numpy())
        # new block: scale = amax / 448 from the token itself, then the same rule
        amax = x[1].abs().amax(dim=-1)
        assert np.array_equal(sc_out[3], (amax / 448.0).numpy())
        r = x[1] / (amax / 448.0)[:, None]
        assert np.array_equal(cache[3, :, 0], r.to(torch.float8_e4m3fn).view(torch.uint8).numpy())
        # nothing else changed
        mask = np.ones(cache.shape, bool)
        mask[1, :, 7] = False
        mask[3, :, 0] = False
        assert np.array_equal(cache[mask], kc.numpy()[mask])


def test_kv_bytes_formula_matches_pages():
    with open(os.path.join(GOLDEN, "kv_bytes_examples.json")) as f:
        ex = json.load(f)["examples"]
    for e in ex:
        total = oracle.kv_bytes_per_token(e["layers"], e["kv_heads"], e["head_dim"],
                                          e["dtype_bytes"]) * e["tokens"]
        if "expect_bytes" in e:
            assert total == e["expect_bytes"], e["what"]
        if "expect_gib_approx" in e:
            assert abs(total / 2 ** 30 - e["expect_gib_approx"]) < 1e-9, e["what"]
        if "expect_gb_approx" in e:
            assert abs(total / 1e9 - e["expect_gb_approx"]) < 0.5, e["what"]


def test_block_table_page_semantics():
    bt = BlockTable(8)
    assert bt.allocate(1, 33)                  # ceil(33/16) = 3 blocks from the end
    assert bt.seq_tables[1] == [7, 6, 5]
    assert not bt.allocate(2, 16 * 6)          # 5 free < 6 needed: OOM, no change
    assert bt.num_free() == 5 and 2 not in bt.seq_tables
    assert bt.fork(1, 2)
    assert [bt.block_refcount[b] for b in (7, 6, 5)] == [2, 2, 2]
    # seq 2 writes token 33 into shared block 5: copy-on-write
    slots, cow = bt.append_slots([2])
    assert cow == [(5, 4)] and slots == [4 * 16 + 1]
    assert bt.seq_tables[2] == [7, 6, 4] and bt.block_refcount[5] == 1
    # seq 1 writes into its (now private) last block: no copy
    slots, cow = bt.append_slots([1])
    assert cow == [] and slots == [5 * 16 + 1]
    bt.free(1)                                  # 7, 6 drop to 1; 5 returns
    assert bt.free_blocks[-1] == 5 and bt.block_refcount[7] == 1
    bt.free(2)
    assert sorted(bt.free_blocks) == list(range(8))


def test_block_table_append_opens_block_and_oom_restores():
    bt = BlockTable(2)
    bt.allocate("a", 16)
    assert bt.append_slots(["a"]) == ([0 * 16 + 0], [])   # free list [0] -> block 0
    assert bt.seq_tables["a"] == [1, 0]
    bt.allocate("b", 0)
    before = (list(bt.free_blocks), dict(bt.seq_tokens))
    assert bt.append_slots(["b"]) is None                  # no free block left
    assert (bt.free_blocks, bt.seq_tokens) == before


def test_block_table_adopt_keeps_free_order():
    bt = BlockTable(6)
    bt.adopt("p", [4, 1], 20)
    bt.adopt("q", [4, 2], 17)
    assert bt.block_refcount[4] == 2
    assert bt.num_free() == 3 and bt.free_blocks == [0, 3, 5]
    slots, cow = bt.append_slots(["p", "q"])
    # p: pos 20 in shared? block 1 (refcount 1) -> no copy; q: pos 17 in block 2
    assert cow == [] and slots == [1 * 16 + 4, 2 * 16 + 1]


def _stream_into_fresh_blocks(calibrated, mags, D=32, Hkv=2, seed=6):
    """Appends len(mags) tokens one call at a time into fresh blocks (token t
    scaled by mags[t]); returns (k cache bytes, k scales, the tokens as fp32)."""
    g = torch.Generator().manual_seed(seed)
    n = len(mags)
    nb = (n + 15) // 16
    kc = np.zeros((nb, Hkv, 16, D), dtype=np.uint8)
    vc = kc.copy()
    ks = np.zeros((nb, Hkv), dtype=np.float32)
    vs = ks.copy()
    toks = (torch.randn((n, Hkv, D), generator=g) * torch.tensor(mags)[:, None, None]).to(torch.bfloat16)
    for t in range(n):
        kc, vc, ks, vs = oracle.append(kc, vc, "fp8_e4m3", toks[t:t + 1], toks[t:t + 1], "bf16", [t],
                                       k_scale=ks, v_scale=vs, calibrated=calibrated)
    return kc, ks, toks.float()


def _pow2_scale(amax):
    """Smallest power of two p with amax <= 448 p (1 for amax 0), from the
    exact search over exponents."""
    out = np.ones_like(amax, dtype=np.float32)
    for i, a in np.ndenumerate(amax):
        if a > 0:
            k = -160
            while float(a) > 448.0 * 2.0 ** k:
                k += 1
            out[i] = np.float32(2.0 ** k)
    return out


def test_calibrated_append_scale_is_the_block_max_power_of_two_and_nothing_saturates():
    """Growing magnitudes ('苦猿的大模型日记 Day45' PART 02: calibration decides
    FP8 quality): every block's scale is the smallest power of two covering
    max|x| / 448 over its tokens, the newest token is the RNE cast of
    x / scale, and every stored value dequantises within one e4m3 rounding
    (2^-4 relative) plus half a subnormal step (2^-10 scale) of its token —
    re-quantisation by a power of two is exact in the normal range.  The
    opener-only rule saturates the same stream."""
    mags = [0.5 * 1.3 ** t for t in range(20)]            # each token larger than the last
    kc, ks, x = _stream_into_fresh_blocks(True, mags)
    xk = x.numpy()
    for blk in range(kc.shape[0]):
        t0, t1 = 16 * blk, min(len(mags), 16 * blk + 16)
        amax = np.abs(xk[t0:t1]).max(axis=(0, 2))               # per kv head
        assert np.array_equal(ks[blk], _pow2_scale(amax))
        last = t1 - 1
        r = torch.from_numpy(xk[last] / ks[blk][:, None])
        assert np.array_equal(kc[blk, :, last - t0], r.to(torch.float8_e4m3fn).view(torch.uint8).numpy())
        deq = torch.from_numpy(kc[blk, :, :t1 - t0]).view(torch.float8_e4m3fn).float().numpy() \
            * ks[blk][:, None, None]
        tru = np.transpose(xk[t0:t1], (1, 0, 2))
        assert np.all(np.abs(deq - tru) <= 2.0 ** -4 * np.abs(tru) + 2.0 ** -10 * ks[blk][:, None, None])
    kc_p, ks_p, _ = _stream_into_fresh_blocks(False, mags)
    deq_p = torch.from_numpy(kc_p[0, :, :16]).view(torch.float8_e4m3fn).float().numpy() * ks_p[0][:, None, None]
    tru = np.transpose(xk[:16], (1, 0, 2))
    assert np.any(np.abs(deq_p - tru) > 0.3 * np.abs(tru))


def test_calibrated_rescale_shifts_exponents_exactly():
    """A token four times larger than the block's first raises the scale by
    2^2; the first token's bytes then dequantise to the same values as
    before whenever they stay in the normal range."""
    base = [1.0, 4.0]
    kc1, ks1, _ = _stream_into_fresh_blocks(True, base[:1], seed=9)
    kc2, ks2, _ = _stream_into_fresh_blocks(True, base, seed=9)
    assert np.all(ks2[0] > ks1[0])
    before = torch.from_numpy(kc1[0, :, 0]).view(torch.float8_e4m3fn).float().numpy() * ks1[0][:, None]
    after = torch.from_numpy(kc2[0, :, 0]).view(torch.float8_e4m3fn).float().numpy() * ks2[0][:, None]
    normal = np.abs(after) >= 2.0 ** -6 * ks2[0][:, None]
    assert normal.sum() > 20 and np.array_equal(before[normal], after[normal])
