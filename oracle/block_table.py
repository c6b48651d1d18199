"""Pure-Python physical-block allocator: the oracle for step a1 (slot mapping
and copy-on-write preparation).  TEST INFRASTRUCTURE ONLY.

Follows the BlockTable of the page "大模型推理加速核心KV Cache 复用机制与内存布局
优化", §三 (PagedAttention: Block Table 管理), whose printed code lost its
operators in extraction.  Readings taken here (each is the only one that makes
the class work):
  * ``self.block_size = block_size``; ``free_blocks = list(range(N))`` and
    blocks are taken with ``pop()``, i.e. from the END of the list (LIFO);
  * allocate(): ``needed = ceil(num_tokens / block_size)``; ``if
    len(free_blocks) < needed: return False`` (the OOM that triggers preemption);
  * fork(): the child's table is a copy of the parent's, each block's refcount
    ``+= 1`` (copy-on-write sharing);
  * free(): refcount ``-= 1`` per block, a block whose count ``== 0`` is
    appended back to the free list;
  * the refcount table (never initialised on the page) starts at 0 and a freshly
    allocated block has count 1.
The write side of copy-on-write is not printed.  Reading: when a sequence
writes a token into a block whose refcount is > 1, it first takes a fresh
block, copies the shared block into it, swaps it into its table and drops one
reference to the old block ("LLM推理优化实战", §2.2: shared prefix blocks are
copied only when a request modifies them).  New tokens go to position
``num_tokens`` ("LLM推理优化实战", §2.2 append_token: logical block =
num_tokens // BLOCK_SIZE); a fresh block is needed only when that position
starts a block.  ``adopt`` (not on the page) registers a table built elsewhere,
removing its blocks from the free list while keeping the order of the rest.

``release_outside_window`` (not on the page; the sliding window / KV eviction
of "苦猿的大模型日记 Day45" PART 02 keeps a fixed cache bound by giving up
history): with window W, the next token (position num_tokens) and every later
one see positions >= num_tokens + 1 - W only, so every block whose 16
positions all lie below that is released — its reference dropped (free list
end when it reaches 0, in table order) and its table entry set to -1.  fork
and free skip -1 entries.
"""


class BlockTable:
    def __init__(self, num_gpu_blocks, block_size=16):
        self.block_size = block_size
        self.num_blocks = num_gpu_blocks
        self.free_blocks = list(range(num_gpu_blocks))
        self.seq_tables = {}
        self.seq_tokens = {}
        self.block_refcount = [0] * num_gpu_blocks
        self._stale = False  # adopted blocks still listed as free

    def _compact(self):
        if self._stale:
            self.free_blocks = [b for b in self.free_blocks if self.block_refcount[b] == 0]
            self._stale = False

    def num_free(self):
        self._compact()
        return len(self.free_blocks)

    def allocate(self, seq_id, num_tokens):
        if seq_id in self.seq_tables or num_tokens < 0:
            raise ValueError("bad allocate")
        self._compact()
        needed = (num_tokens + self.block_size - 1) // self.block_size
        if len(self.free_blocks) < needed:
            return False
        allocated = [self.free_blocks.pop() for _ in range(needed)]
        for blk in allocated:
            self.block_refcount[blk] = 1
        self.seq_tables[seq_id] = allocated
        self.seq_tokens[seq_id] = num_tokens
        return True

    def adopt(self, seq_id, blocks, num_tokens):
        if seq_id in self.seq_tables:
            raise ValueError("sequence exists")
        if len(blocks) != (num_tokens + self.block_size - 1) // self.block_size:
            raise ValueError("table length does not match num_tokens")
        for blk in blocks:
            if not 0 <= blk < self.num_blocks:
                raise ValueError("block id out of range")
        for blk in blocks:
            self.block_refcount[blk] += 1
        self._stale = True
        self.seq_tables[seq_id] = list(blocks)
        self.seq_tokens[seq_id] = num_tokens

    def fork(self, parent_id, child_id):
        if parent_id not in self.seq_tables or child_id in self.seq_tables:
            return False
        parent_blocks = self.seq_tables[parent_id]
        self.seq_tables[child_id] = list(parent_blocks)
        self.seq_tokens[child_id] = self.seq_tokens[parent_id]
        for blk in parent_blocks:
            if blk >= 0:
                self.block_refcount[blk] += 1
        return True

    def free(self, seq_id):
        self._compact()
        for blk in self.seq_tables[seq_id]:
            if blk < 0:
                continue
            self.block_refcount[blk] -= 1
            if self.block_refcount[blk] == 0:
                self.free_blocks.append(blk)
        del self.seq_tables[seq_id]
        del self.seq_tokens[seq_id]

    def release_outside_window(self, seq_id, window):
        """Releases the blocks no later token can see; returns how many."""
        if window < 1:
            raise ValueError("window must be >= 1")
        self._compact()
        table = self.seq_tables[seq_id]
        first_visible = self.seq_tokens[seq_id] + 1 - window
        n = min(len(table), max(0, first_visible) // self.block_size)
        released = 0
        for j in range(n):
            blk = table[j]
            if blk < 0:
                continue
            self.block_refcount[blk] -= 1
            if self.block_refcount[blk] == 0:
                self.free_blocks.append(blk)
            table[j] = -1
            released += 1
        return released

    def append_slots(self, seq_ids):
        """One new token per sequence.  Returns (slots, cow_pairs) or None on
        OOM, in which case nothing has changed."""
        self._compact()
        saved = (list(self.free_blocks), {s: list(t) for s, t in self.seq_tables.items()},
                 dict(self.seq_tokens), list(self.block_refcount))
        slots, cow = [], []
        for seq in seq_ids:
            table = self.seq_tables[seq]
            pos = self.seq_tokens[seq]
            logical = pos // self.block_size
            if pos % self.block_size == 0:
                if not self.free_blocks:
                    self._restore(saved)
                    return None
                blk = self.free_blocks.pop()
                self.block_refcount[blk] = 1
                table.append(blk)
            else:
                old = table[logical]
                if self.block_refcount[old] > 1:
                    if not self.free_blocks:
                        self._restore(saved)
                        return None
                    new = self.free_blocks.pop()
                    self.block_refcount[new] = 1
                    self.block_refcount[old] -= 1
                    table[logical] = new
                    cow.append((old, new))
            slots.append(table[logical] * self.block_size + pos % self.block_size)
            self.seq_tokens[seq] = pos + 1
        return slots, cow

    def _restore(self, saved):
        self.free_blocks, self.seq_tables, self.seq_tokens, self.block_refcount = saved
