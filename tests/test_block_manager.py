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
        elif op < 0.6:
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
