// block_manager.cpp — step a1 on the host: physical-block allocation, fork,
// free and the per-token slot mapping with copy-on-write.
//
// Semantics follow the BlockTable of "大模型推理加速核心KV Cache 复用机制与内存
// 布局优化" §三: a free list that starts as [0..N-1] and hands out blocks from
// its end; allocate takes ceil(n / 16) blocks or fails unchanged; fork shares
// the parent's blocks and raises their reference counts; free lowers them and
// returns blocks that reach zero to the end of the free list.  The write side
// of copy-on-write ("LLM推理优化实战" §2.2: shared blocks are copied only when a
// request modifies them) swaps a fresh block into the writer's table before a
// token lands in a block whose count is above one.
#include <stdint.h>

#include <algorithm>
#include <new>
#include <unordered_map>
#include <vector>

#include "pagedkv.h"

struct pkv_block_manager {
  int64_t num_blocks = 0;
  std::vector<int32_t> free_list;     // taken from the back
  std::vector<int32_t> refcount;
  bool stale = false;                 // adopted blocks still listed as free
  struct Seq {
    std::vector<int32_t> table;
    int64_t tokens = 0;
  };
  std::unordered_map<int64_t, Seq> seqs;

  void compact() {
    if (!stale) return;
    size_t k = 0;
    for (size_t i = 0; i < free_list.size(); ++i)
      if (refcount[free_list[i]] == 0) free_list[k++] = free_list[i];
    free_list.resize(k);
    stale = false;
  }
};

namespace {
constexpr int64_t kBS = PKV_BLOCK_SIZE;
inline int64_t blocks_for(int64_t tokens) { return (tokens + kBS - 1) / kBS; }
}  // namespace

extern "C" {

pkv_block_manager *pkv_bm_create(int64_t num_blocks) {
  if (num_blocks <= 0 || num_blocks > INT32_MAX) return nullptr;
  pkv_block_manager *bm = new (std::nothrow) pkv_block_manager();
  if (!bm) return nullptr;
  try {
    bm->num_blocks = num_blocks;
    bm->free_list.resize((size_t)num_blocks);
    for (int64_t i = 0; i < num_blocks; ++i) bm->free_list[(size_t)i] = (int32_t)i;
    bm->refcount.assign((size_t)num_blocks, 0);
  } catch (...) {
    delete bm;
    return nullptr;
  }
  return bm;
}

void pkv_bm_destroy(pkv_block_manager *bm) { delete bm; }

int pkv_bm_allocate(pkv_block_manager *bm, int64_t seq, int64_t num_tokens) {
  if (!bm || num_tokens < 0 || bm->seqs.count(seq)) return PKV_EINVAL;
  bm->compact();
  const int64_t needed = blocks_for(num_tokens);
  if ((int64_t)bm->free_list.size() < needed) return PKV_EOOM;
  pkv_block_manager::Seq s;
  s.tokens = num_tokens;
  s.table.reserve((size_t)needed);
  for (int64_t i = 0; i < needed; ++i) {
    const int32_t blk = bm->free_list.back();
    bm->free_list.pop_back();
    bm->refcount[blk] = 1;
    s.table.push_back(blk);
  }
  bm->seqs.emplace(seq, std::move(s));
  return PKV_OK;
}

int pkv_bm_adopt(pkv_block_manager *bm, int64_t seq, const int32_t *blocks, int nblocks, int64_t num_tokens) {
  if (!bm || num_tokens < 0 || nblocks < 0 || (nblocks > 0 && !blocks) || bm->seqs.count(seq)) return PKV_EINVAL;
  if (blocks_for(num_tokens) != nblocks) return PKV_EINVAL;
  for (int i = 0; i < nblocks; ++i)
    if (blocks[i] < 0 || blocks[i] >= bm->num_blocks) return PKV_ERANGE;
  pkv_block_manager::Seq s;
  s.tokens = num_tokens;
  s.table.assign(blocks, blocks + nblocks);
  for (int i = 0; i < nblocks; ++i) bm->refcount[blocks[i]] += 1;
  bm->stale = bm->stale || nblocks > 0;
  bm->seqs.emplace(seq, std::move(s));
  return PKV_OK;
}

int pkv_bm_fork(pkv_block_manager *bm, int64_t parent, int64_t child) {
  if (!bm) return PKV_EINVAL;
  auto it = bm->seqs.find(parent);
  if (it == bm->seqs.end()) return PKV_ENOTFOUND;
  if (bm->seqs.count(child)) return PKV_EINVAL;
  pkv_block_manager::Seq s = it->second;
  for (int32_t blk : s.table)
    if (blk >= 0) bm->refcount[blk] += 1;
  bm->seqs.emplace(child, std::move(s));
  return PKV_OK;
}

int pkv_bm_free(pkv_block_manager *bm, int64_t seq) {
  if (!bm) return PKV_EINVAL;
  auto it = bm->seqs.find(seq);
  if (it == bm->seqs.end()) return PKV_ENOTFOUND;
  bm->compact();
  for (int32_t blk : it->second.table)
    if (blk >= 0 && --bm->refcount[blk] == 0) bm->free_list.push_back(blk);
  bm->seqs.erase(it);
  return PKV_OK;
}

int pkv_bm_release_window(pkv_block_manager *bm, int64_t seq, int64_t window, int64_t *released_out) {
  if (!bm || window < 1) return PKV_EINVAL;
  auto it = bm->seqs.find(seq);
  if (it == bm->seqs.end()) return PKV_ENOTFOUND;
  bm->compact();
  std::vector<int32_t> &table = it->second.table;
  const int64_t first_visible = it->second.tokens + 1 - window;
  const int64_t n = std::min<int64_t>((int64_t)table.size(), first_visible > 0 ? first_visible / kBS : 0);
  int64_t released = 0;
  for (int64_t j = 0; j < n; ++j) {
    const int32_t blk = table[(size_t)j];
    if (blk < 0) continue;
    if (--bm->refcount[blk] == 0) bm->free_list.push_back(blk);
    table[(size_t)j] = -1;
    ++released;
  }
  if (released_out) *released_out = released;
  return PKV_OK;
}

int pkv_bm_append_slots(pkv_block_manager *bm, const int64_t *seqs, int n, int64_t *slot_out, int32_t *cow_pairs_out,
                        int *n_cow_out) {
  if (!bm || n < 0 || (n > 0 && (!seqs || !slot_out || !cow_pairs_out)) || !n_cow_out) return PKV_EINVAL;
  bm->compact();
  // all sequences must exist before anything changes
  for (int i = 0; i < n; ++i)
    if (!bm->seqs.count(seqs[i])) return PKV_ENOTFOUND;
  struct Undo {
    int64_t seq;
    int64_t tokens;
    bool appended;      // a block was pushed to the table
    int64_t logical;    // table index replaced by copy-on-write (-1 if none)
    int32_t old_blk;
  };
  std::vector<Undo> undo;
  std::vector<int32_t> taken;
  undo.reserve((size_t)n);
  int ncow = 0;
  bool oom = false;
  for (int i = 0; i < n && !oom; ++i) {
    pkv_block_manager::Seq &s = bm->seqs[seqs[i]];
    const int64_t pos = s.tokens;
    const int64_t logical = pos / kBS;
    Undo u{seqs[i], s.tokens, false, -1, -1};
    if (pos % kBS == 0) {
      if (bm->free_list.empty()) { oom = true; break; }
      const int32_t blk = bm->free_list.back();
      bm->free_list.pop_back();
      taken.push_back(blk);
      bm->refcount[blk] = 1;
      s.table.push_back(blk);
      u.appended = true;
    } else {
      const int32_t old = s.table[(size_t)logical];
      if (bm->refcount[old] > 1) {
        if (bm->free_list.empty()) { oom = true; break; }
        const int32_t blk = bm->free_list.back();
        bm->free_list.pop_back();
        taken.push_back(blk);
        bm->refcount[blk] = 1;
        bm->refcount[old] -= 1;
        s.table[(size_t)logical] = blk;
        u.logical = logical;
        u.old_blk = old;
        cow_pairs_out[2 * ncow] = old;
        cow_pairs_out[2 * ncow + 1] = blk;
        ++ncow;
      }
    }
    slot_out[i] = (int64_t)s.table[(size_t)logical] * kBS + pos % kBS;
    s.tokens = pos + 1;
    undo.push_back(u);
  }
  if (oom) {  // roll back in reverse order; taken blocks return in reverse pop order
    for (size_t k = undo.size(); k-- > 0;) {
      const Undo &u = undo[k];
      pkv_block_manager::Seq &s = bm->seqs[u.seq];
      s.tokens = u.tokens;
      if (u.appended) {
        bm->refcount[s.table.back()] = 0;
        s.table.pop_back();
      } else if (u.logical >= 0) {
        bm->refcount[s.table[(size_t)u.logical]] = 0;
        s.table[(size_t)u.logical] = u.old_blk;
        bm->refcount[u.old_blk] += 1;
      }
    }
    for (size_t k = taken.size(); k-- > 0;) bm->free_list.push_back(taken[k]);
    *n_cow_out = 0;
    return PKV_EOOM;
  }
  *n_cow_out = ncow;
  return PKV_OK;
}

int pkv_bm_export(const pkv_block_manager *bm, const int64_t *seqs, int n, int32_t *table_out, int max_blocks,
                  int32_t *context_lens_out) {
  if (!bm || n < 0 || max_blocks <= 0 || (n > 0 && (!seqs || !table_out || !context_lens_out))) return PKV_EINVAL;
  for (int i = 0; i < n; ++i) {
    auto it = bm->seqs.find(seqs[i]);
    if (it == bm->seqs.end()) return PKV_ENOTFOUND;
    if ((int64_t)it->second.table.size() > max_blocks || it->second.tokens > INT32_MAX) return PKV_ERANGE;
  }
  for (int i = 0; i < n; ++i) {
    const pkv_block_manager::Seq &s = bm->seqs.at(seqs[i]);
    int32_t *row = table_out + (size_t)i * max_blocks;
    size_t j = 0;
    for (; j < s.table.size(); ++j) row[j] = s.table[j];
    for (; j < (size_t)max_blocks; ++j) row[j] = -1;
    context_lens_out[i] = (int32_t)s.tokens;
  }
  return PKV_OK;
}

int64_t pkv_bm_num_free(const pkv_block_manager *bm) {
  if (!bm) return -1;
  if (!bm->stale) return (int64_t)bm->free_list.size();
  int64_t n = 0;
  for (int32_t b : bm->free_list)
    if (bm->refcount[b] == 0) ++n;
  return n;
}

int pkv_bm_refcount(const pkv_block_manager *bm, int64_t block) {
  if (!bm || block < 0 || block >= bm->num_blocks) return -1;
  return bm->refcount[(size_t)block];
}

int64_t pkv_bm_num_tokens(const pkv_block_manager *bm, int64_t seq) {
  if (!bm) return -1;
  auto it = bm->seqs.find(seq);
  return it == bm->seqs.end() ? -1 : it->second.tokens;
}

}  // extern "C"
