"""Pins of the oracle's block table (step a1) that involve no native code:
sliding-window release against its closed form, and planted mistakes in a
copy of oracle/block_table.py that the pins must catch.  Host only.

Window release ("苦猿的大模型日记 Day45" PART 02, sliding window / KV eviction:
a fixed visible history bounds the cache).  The next token of a sequence
holding `tokens` positions sits at position `tokens`; with window W it and
every later token see positions >= tokens + 1 - W, so exactly the logical
blocks j with 16 (j + 1) <= tokens + 1 - W can go: max(0, tokens + 1 - W) // 16
of them.  With q_len new tokens per step the step's first token is the one at
position `tokens`, so the same count holds before each step's reservation.
"""
import importlib.util

import pytest

import test_oracle_append_and_formula as T_app
from oracle import block_table as _bt_module

BlockTable = _bt_module.BlockTable
BLOCK = 16


def _released_prefix(table):
    n = 0
    while n < len(table) and table[n] == -1:
        n += 1
    return n


@pytest.mark.parametrize("W", [1, 16, 17, 40])
@pytest.mark.parametrize("q_len", [1, 4])
@pytest.mark.parametrize("start", [0, 3, 16])
def test_window_release_matches_closed_form(W, q_len, start):
    """Decode one sequence for 160 tokens, releasing before each step:
    released entries = max(0, tokens + 1 - W) // 16 (never more than the table
    holds), only a prefix of the table is released, every released block lies
    wholly before the window and the first kept one does not, and the free
    list gets exactly the released blocks back."""
    N = 64
    bt = BlockTable(N)
    assert bt.allocate(0, start)
    total_released = 0
    while bt.seq_tokens[0] < start + 160:
        tokens = bt.seq_tokens[0]
        table = bt.seq_tables[0]
        before = _released_prefix(table)
        got = bt.release_outside_window(0, W)
        want = min(len(table), max(0, tokens + 1 - W) // BLOCK)
        n = _released_prefix(table)
        assert n == want, (tokens, W, n, want)
        assert got == want - before                       # only newly released entries count
        assert all(b >= 0 for b in table[n:])             # released entries form a prefix
        first_visible = tokens + 1 - W
        assert all(BLOCK * (j + 1) <= first_visible for j in range(n))
        if n < len(table):
            assert BLOCK * (n + 1) > first_visible        # the first kept block reaches the window
        total_released += got
        held = sum(1 for b in table if b >= 0)
        assert bt.num_free() == N - held
        slots, cow = bt.append_slots([0] * q_len)
        assert cow == []
        assert [s % BLOCK for s in slots] == [(tokens + t) % BLOCK for t in range(q_len)]
        # a sequence never holds more than ceil((W + q_len - 1) / 16) + 1 blocks
        held = sum(1 for b in bt.seq_tables[0] if b >= 0)
        assert held <= -(-(W + q_len - 1) // BLOCK) + 1
    assert total_released == _released_prefix(bt.seq_tables[0])


def test_window_release_order_and_shared_blocks():
    """Released blocks go back to the END of the free list in table order,
    so the next block taken is the last one released (LIFO); a block another
    sequence still references loses one reference and stays allocated."""
    bt = BlockTable(8)
    assert bt.allocate(0, 48)                   # blocks 7, 6, 5
    assert bt.seq_tables[0] == [7, 6, 5]
    assert bt.allocate(2, 20)                   # blocks 4, 3; free list [0, 1, 2]
    assert bt.release_outside_window(2, 4) == 1  # 20 + 1 - 4 = 17: logical block 0 (id 4)
    assert bt.seq_tables[2] == [-1, 3] and bt.free_blocks == [0, 1, 2, 4]
    assert bt.allocate(3, 1) and bt.seq_tables[3] == [4]   # the last released is taken first
    bt.free(3)
    bt.free(2)                                  # the -1 entry is skipped
    assert bt.free_blocks == [0, 1, 2, 4, 3]
    assert bt.fork(0, 1)
    assert bt.release_outside_window(0, 1) == 3  # 48 + 1 - 1 = 48: all three blocks
    assert bt.seq_tables[0] == [-1, -1, -1]
    assert [bt.block_refcount[b] for b in (7, 6, 5)] == [1, 1, 1]
    assert bt.num_free() == 5                    # still referenced by sequence 1
    bt.free(1)
    assert bt.free_blocks[-3:] == [7, 6, 5]      # table order
    slots, _ = bt.append_slots([0])              # position 48 opens a block: takes 5
    assert slots == [5 * BLOCK + 0]
    assert bt.release_outside_window(0, 1) == 0  # 49 + 1 - 1 = 49: block 3 of 4 still visible
    with pytest.raises(ValueError):
        bt.release_outside_window(0, 0)


def test_window_release_special_cases():
    bt = BlockTable(8)
    assert bt.allocate(0, 15)
    assert bt.release_outside_window(0, 1) == 0   # 15 + 1 - 1 = 15 < 16: nothing to drop
    bt.append_slots([0])                          # 16 tokens
    assert bt.release_outside_window(0, 1) == 1   # 16 + 1 - 1 = 16: block 0 wholly before
    bt2 = BlockTable(8)
    assert bt2.allocate(0, 64)                    # 4 blocks
    assert bt2.release_outside_window(0, 1 << 20) == 0   # a window wider than the sequence


# ---------------------------------------------------------------------------
# Planted mistakes in a copy of oracle/block_table.py: each must fail a pin
# above or in test_oracle_append_and_formula (none of them involves the
# native block manager).
# ---------------------------------------------------------------------------
_SRC = _bt_module.__file__

_release_pins = [lambda: test_window_release_matches_closed_form(17, 1, 3),
                 lambda: test_window_release_matches_closed_form(16, 4, 3),
                 test_window_release_special_cases]

MUTANTS = [
    ("release one block too many",
     "n = min(len(table), max(0, first_visible) // self.block_size)",
     "n = min(len(table), max(0, first_visible) // self.block_size + 1)", _release_pins),
    ("release one block too few",
     "n = min(len(table), max(0, first_visible) // self.block_size)",
     "n = min(len(table), max(0, first_visible - self.block_size) // self.block_size)", _release_pins),
    ("window start without the next token",
     "first_visible = self.seq_tokens[seq_id] + 1 - window",
     "first_visible = self.seq_tokens[seq_id] - window", _release_pins),
    ("free list taken from the front",
     "allocated = [self.free_blocks.pop() for _ in range(needed)]",
     "allocated = [self.free_blocks.pop(0) for _ in range(needed)]",
     [T_app.test_block_table_page_semantics]),
    ("floor instead of ceil in allocate",
     "needed = (num_tokens + self.block_size - 1) // self.block_size",
     "needed = num_tokens // self.block_size",
     [T_app.test_block_table_page_semantics]),
    ("copy on write of a private block",
     "if self.block_refcount[old] > 1:",
     "if self.block_refcount[old] >= 1:",
     [T_app.test_block_table_page_semantics, T_app.test_block_table_adopt_keeps_free_order]),
    ("released blocks not returned",
     "            if self.block_refcount[blk] == 0:\n                self.free_blocks.append(blk)\n            table[j] = -1",
     "            table[j] = -1",
     [test_window_release_order_and_shared_blocks,
      lambda: test_window_release_matches_closed_form(40, 1, 0)]),
]


@pytest.mark.parametrize("name,orig,mut,tests", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_block_table_mistake_is_caught(tmp_path, monkeypatch, name, orig, mut, tests):
    with open(_SRC) as f:
        src = f.read()
    assert src.count(orig) == 1, f"fragment for '{name}' not unique in block_table.py"
    path = tmp_path / "block_table_mutant.py"
    path.write_text(src.replace(orig, mut))
    spec = importlib.util.spec_from_file_location("block_table_mutant", str(path))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    monkeypatch.setattr(T_app, "BlockTable", mod.BlockTable)
    monkeypatch.setitem(globals(), "BlockTable", mod.BlockTable)
    caught = 0
    for t in tests:
        try:
            t()
        except (AssertionError, ValueError, IndexError, TypeError):
            caught += 1
    assert caught == len(tests), f"mutant '{name}' survived its pin tests"
