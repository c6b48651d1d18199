"""The native block manager (step a1, in libpagedkv.so) against the oracle's
pure-Python BlockTable on random operation sequences: identical block ids,
refcounts, slots and copy-on-write pairs.  Host only."""
import random

import numpy as np
import pytest

from oracle.block_table import BlockTable


def _pkv():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_gqa_03_gb300 as pkv
    return pkv


@pytest.mark.parametrize("seed", range(6))
def test_native_matches_oracle_on_random_ops(seed):
    pkv = _pkv()
    rng = random.Random(seed)
    N = rng.choice([8, 40, 200])
    ref, bm = BlockTable(N), pkv.BlockManager(N)
    live, next_id = [], 0
    for _ in range(400):
        op = rng.random()
        if op < 0.25 or not live:
            n = rng.randrange(0, 60)
            a, b = ref.allocate(next_id, n), bm.allocate(next_id, n)
            assert a == b
            if a:
                live.append(next_id)
            next_id += 1
        elif op < 0.4:
            p = rng.choice(live)
            assert ref.fork(p, next_id) == bm.fork(p, next_id)
            live.append(next_id)
            next_id += 1
        elif op < 0.55:
            s = live.pop(rng.randrange(len(live)))
            ref.free(s)
            bm.free(s)
        elif op < 0.62 and live:
            s = rng.choice(live)
            w = rng.randrange(1, 50)
            assert ref.release_outside_window(s, w) == bm.release_outside_window(s, w)
        elif op < 0.67:
            blocks = rng.sample(range(N), rng.randrange(0, 4))
            ntok = len(blocks) * 16 - rng.randrange(0, 16) if blocks else 0
            ref.adopt(next_id, blocks, ntok)
            bm.adopt(next_id, blocks, ntok)
            live.append(next_id)
            next_id += 1
        else:
            seqs = rng.sample(live, rng.randrange(1, min(len(live), 5) + 1))
            r, n = ref.append_slots(seqs), bm.append_slots(seqs)
            assert r == (None if n is None else (n[0], n[1]))
        assert ref.num_free() == bm.num_free()
        if live:
            mb = max(1, max(len(ref.seq_tables[s]) for s in live))
            table, lens = bm.export(live, mb)
            for i, s in enumerate(live):
                t = ref.seq_tables[s]
                assert list(table[i, :len(t)]) == t and all(table[i, len(t):] == -1)
                assert lens[i] == ref.seq_tokens[s]
        for blk in range(N):
            assert ref.block_refcount[blk] == bm.refcount(blk)


def test_release_outside_window_bounds_the_cache():
    """Decoding one sequence for 400 tokens with window 40 keeps at most
    ceil(40 / 16) + 1 blocks; a fork shares the kept blocks only."""
    pkv = _pkv()
    bm, ref = pkv.BlockManager(64), BlockTable(64)
    for m in (bm, ref):
        assert m.allocate(0, 5)
    for step in range(400):
        assert bm.release_outside_window(0, 40) == ref.release_outside_window(0, 40)
        assert bm.append_slots([0]) == ref.append_slots([0])
        table, lens = bm.export([0], 64)
        held = [b for b in table[0] if b >= 0]
        assert len(held) <= 4 and bm.num_free() == 64 - len(held)
        assert list(table[0, :len(ref.seq_tables[0])]) == ref.seq_tables[0]
    first = (int(lens[0]) - 40) // 16                 # released logical blocks stay -1
    assert all(table[0, :first] == -1)
    assert bm.fork(0, 1) and ref.fork(0, 1)
    for blk in held:
        assert bm.refcount(blk) == 2 == ref.block_refcount[blk]
    bm.free(0), ref.free(0), bm.free(1), ref.free(1)
    assert bm.num_free() == 64 == ref.num_free()
    with pytest.raises(pkv.PagedKVError):
        bm.release_outside_window(5, 40)            # unknown sequence
    assert bm.allocate(5, 1)
    with pytest.raises(pkv.PagedKVError):
        bm.release_outside_window(5, 0)             # window must be >= 1


def test_errors():
    pkv = _pkv()
    bm = pkv.BlockManager(4)
    assert bm.allocate(1, 16)
    with pytest.raises(pkv.PagedKVError):
        bm.allocate(1, 16)                      # duplicate id
    assert not bm.fork(7, 8)                    # unknown parent
    with pytest.raises(pkv.PagedKVError):
        bm.adopt(2, [9], 5)                     # block out of range
    with pytest.raises(pkv.PagedKVError):
        bm.adopt(2, [0, 1], 5)                  # table longer than ceil(5/16)
    with pytest.raises(pkv.PagedKVError):
        bm.append_slots([42])                   # unknown sequence
    assert not bm.allocate(3, 16 * 4)           # OOM leaves everything unchanged
    assert bm.num_free() == 3
