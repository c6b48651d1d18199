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
