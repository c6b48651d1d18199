// prefill.cu — paged prefill attention on the fifth-generation tensor cores
// (tcgen05): every new token of a sequence attends causally to the sequence's
// paged cache (its prompt and any cached prefix), optionally inside a sliding
// window.
//
// The computation is FlashAttention's tiled form ("LLM推理优化实战" §3.2
// flash_attention: Q in row blocks, K / V in blocks of 128 positions, online
// softmax with running max m and sum l, O rescaled by exp(m_old - m_new)) with
// the causal mask of "苦猿的大模型日记 Day45" PART 04.  GB300 design:
//  * work items of (sequence, kv head, tile of 128 query rows); a row is (new
//    token i, query head g) of the kv head's group, token-major, so GQA heads
//    share every K / V tile;
//  * one persistent CTA per SM walks its items round by round, the items
//    ordered heaviest first and dealt out serpentine so the CTAs' totals stay
//    near the mean; tensor memory, barriers and the K / V pipeline live
//    across items, so an item's epilogue overlaps the next item's loads and S
//    MMAs, and the next item's Q is copied asynchronously during the current
//    item's last tile (prefill_tiles.cu runs one CTA per item instead);
//  * the tile pipeline (K / V rings, S / P / O in tensor memory, softmax
//    warps, warp roles) is the one described in prefill_common.cuh.
#include "prefill.h"
#include "prefill_common.cuh"

namespace pkv {

// One work item: (row tile, kv head, sequence); every role derives the same
// description from the item index.
struct PrefillItem {
  int b, h, qs, n, R, r0, ctx, nblk, first, j_first, T;
  bool valid;  // the tile holds rows of the sequence
  bool bad_q;  // the sequence's new-token count is negative or above max_q_len (flagged once)
  bool bad_ctx;
};

template <class Cfg>
__device__ __forceinline__ PrefillItem prefill_item(const PrefillParams &p, int i) {
  PrefillItem it;
  // heaviest (latest) row tiles first: the rank over (sequence, kv head) varies fastest
  const int per_rank = p.B * p.Hkv;
  const int tile = p.max_tiles - 1 - i / per_rank;
  const int rest = i % per_rank;
  it.b = rest / p.Hkv;
  it.h = rest % p.Hkv;
  it.qs = p.q_start ? __ldg(p.q_start + it.b) : it.b * p.uniform_q_len;
  it.n = p.q_start ? __ldg(p.q_start + it.b + 1) - it.qs : p.uniform_q_len;
  it.bad_q = tile == 0 && (it.n > p.max_q_len || it.n < 0);
  it.R = it.n * p.G;
  it.r0 = tile * Cfg::M;
  it.valid = it.n > 0 && it.r0 < it.R;
  const int ctx_raw = __ldg(p.context_lens + it.b);
  it.ctx = ctx_raw < 0 ? 0 : (ctx_raw > p.max_blocks * kBlock ? p.max_blocks * kBlock : ctx_raw);
  it.bad_ctx = it.valid && ctx_raw != it.ctx;
  it.nblk = (it.ctx + kBlock - 1) / kBlock;
  it.first = it.j_first = it.T = 0;
  if (it.valid) {
    const int i_lo = it.r0 / p.G, i_hi = min(it.R - 1, it.r0 + Cfg::M - 1) / p.G;
    const int lim_lo = it.ctx - it.n + i_lo + 1, lim_hi = it.ctx - it.n + i_hi + 1;  // exclusive causal ends
    it.first = p.window > 0 ? max(0, lim_lo - p.window) : 0;
    it.j_first = it.first / Cfg::N;
    it.T = lim_hi > 0 ? (lim_hi - 1) / Cfg::N - it.j_first + 1 : 0;  // K / V tiles to stream
  }
  return it;
}

// The CTA's item of round k: rounds deal the items out serpentine (CTA c
// takes k * grid + c in even rounds, k * grid + grid - 1 - c in odd ones), so
// with the items ordered heaviest first the CTAs' totals stay near the mean.
// May be past the item count in the last round.
__device__ __forceinline__ int round_item(int k) {
  const int c = (int)blockIdx.x, G = (int)gridDim.x;
  return k * G + ((k & 1) ? G - 1 - c : c);
}

// Shared memory the persistent kernel's epilogue stages output rows in
// (store_rows_staged): 2 KiB per softmax warp.
constexpr int kOutStage = 8 * 2048;

// Persistent: one CTA per SM walks its work items round by round; tensor
// memory, barriers and the K / V pipeline live across items, so one item's
// epilogue overlaps the next item's loads and S MMAs.
template <class Cfg>
__global__ void __launch_bounds__(Cfg::THREADS, 1)
    prefill_kernel(const __grid_constant__ PrefillParams p, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t *sQ = smem;
  uint8_t *sK = sQ + Cfg::Q_BYTES;
  uint8_t *sV = sK + (size_t)Cfg::KSTAGES * Cfg::KV_BYTES;
  uint8_t *sO = sV + (size_t)Cfg::VSTAGES * Cfg::KV_BYTES;  // epilogue staging, kOutStage bytes
  __shared__ __align__(8) uint64_t k_full[Cfg::KSTAGES], k_empty[Cfg::KSTAGES];
  __shared__ __align__(8) uint64_t v_full[Cfg::VSTAGES], v_empty[Cfg::VSTAGES];
  // per S buffer: S written, P written, P . V done.  (One P barrier per buffer:
  // the softmax may finish tile g + 1 before the MMA warp waits for tile g, but
  // it cannot finish tile g + SBUF before that.)
  __shared__ __align__(8) uint64_t s_full[Cfg::SBUF], p_full[Cfg::SBUF], pv_done[Cfg::SBUF];
  // per item: Q staged, O read out; per pair of softmax warps holding the same
  // rows (w, w + 4): row-max exchange per tile, row-sum exchange per item
  __shared__ __align__(8) uint64_t q_full, o_free, fin;
  __shared__ __align__(8) uint64_t xch[Cfg::SOFTMAX / 64][2], xl[Cfg::SOFTMAX / 64];
  static_assert(Cfg::SOFTMAX / 64 == 4, "four pairs of softmax warps (w, w + 4)");
  __shared__ __align__(8) uint64_t dead;
  __shared__ float red[2][2][Cfg::M];  // partial row maxima [tile parity][half][row]
  __shared__ float red_l[2][Cfg::M];   // partial row sums [half][row]
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag, cta_flags, k_consumed, v_consumed, k_issued, v_issued;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_items = p.max_tiles * p.Hkv * p.B;
  const int n_rounds = (n_items + (int)gridDim.x - 1) / (int)gridDim.x;

  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < Cfg::KSTAGES; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
#pragma unroll
    for (int s = 0; s < Cfg::VSTAGES; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
#pragma unroll
    for (int s = 0; s < Cfg::SBUF; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&p_full[s], Cfg::SOFTMAX / 32);
      mbar_init(&pv_done[s], 1);
    }
    mbar_init(&q_full, Cfg::SOFTMAX / 32);
    mbar_init(&o_free, Cfg::SOFTMAX / 32);
#pragma unroll
    for (int pr = 0; pr < Cfg::SOFTMAX / 64; ++pr) {
      mbar_init(&xch[pr][0], 2);
      mbar_init(&xch[pr][1], 2);
      mbar_init(&xl[pr], 2);
    }
    mbar_init(&fin, 2);  // one commit from each issuing warp
    mbar_init(&dead, 1);  // failure-path test hook: nothing ever arrives on it
    fence_barrier_init();
    abort_flag = 0;
    cta_flags = 0;
    k_consumed = v_consumed = k_issued = v_issued = 0;
  }
  if (warp == Cfg::ISSUER) tc::alloc(&tmem_base, Cfg::TMEM_COLS);
  if (warp == Cfg::PRODUCER && lane == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tbase = tmem_base;

  if (warp == Cfg::PRODUCER || warp == Cfg::V_PRODUCER) {
    // ---------------- TMA producers: every K tile (warp 8) / V tile (warp 10) of every item ----------------
    // lane l fetches block (l % 8) of a tile, panel l / 8; a cursor walks the
    // CTA's tiles across items, fetching block ids three tiles ahead
    const int slot = lane & (Cfg::BLOCKS - 1), panel = lane / Cfg::BLOCKS;
    int ck = -1, cj = 0, cT = 0;  // cursor: tile cj of the cT of round ck's item
    PrefillItem ct{};
    auto step = [&]() -> bool {  // to the cursor's next tile; false past the CTA's last
      if (++cj < cT) return true;
      for (++ck; ck < n_rounds; ++ck) {
        const int ci = round_item(ck);
        if (ci >= n_items) continue;
        ct = prefill_item<Cfg>(p, ci);
        if (ct.valid && ct.T > 0) {
          cj = 0;
          cT = ct.T;
          return true;
        }
      }
      return false;
    };
    int bad = 0;
    // this lane's block of the cursor tile: its raw id, loaded here and first
    // used when the tile's copies are issued (three tiles on), so the load's
    // latency is hidden; none = past the context, or wholly before every
    // row's window (such blocks may have been released)
    struct Pend {
      int id, h;
      bool none;
    };
    auto fetch = [&]() -> Pend {
      Pend f;
      const int lb = (ct.j_first + cj) * Cfg::BLOCKS + slot;
      f.h = ct.h;
      f.none = lb >= ct.nblk || (lb + 1) * kBlock <= ct.first;
      f.id = f.none ? 0 : __ldg(p.block_table + (size_t)ct.b * p.max_blocks + lb);
      return f;
    };
    // the box row of a fetched block: the box past the tensor (zeros) for none
    // or a bad id
    auto row_of = [&](const Pend &f) -> int64_t {
      if (f.none) return p.num_blocks * p.Hkv;
      const bool good = f.id >= 0 && (int64_t)f.id < p.num_blocks;
      bad |= good ? 0 : 1;
      return good ? (int64_t)f.id * p.Hkv + f.h : p.num_blocks * p.Hkv;
    };
    auto issue_k = [&](int g, int64_t trow) -> bool {
      const int ks = g % Cfg::KSTAGES;
      if (g >= Cfg::KSTAGES && !warp_wait(&k_empty[ks], (uint32_t)((g / Cfg::KSTAGES) - 1) & 1u, p.timeout_ns))
        return false;
      if (__any_sync(kFull, *(volatile int *)&abort_flag)) return false;
      if (lane == 0) mbar_arrive_expect_tx(&k_full[ks], Cfg::KV_BYTES);
      __syncwarp();
      if (lane < Cfg::LOADS)
        tma_load_2d(sK + (size_t)ks * Cfg::KV_BYTES + panel * Cfg::PANEL_KV + slot * 2048, &tmK, panel * 64,
                    (int)(trow * kBlock), &k_full[ks]);
      if (lane == 0) k_issued = g + 1;
      return true;
    };
    auto issue_v = [&](int g, int64_t trow) -> bool {
      const int vs = g % Cfg::VSTAGES;
      if (g >= Cfg::VSTAGES && !warp_wait(&v_empty[vs], (uint32_t)((g / Cfg::VSTAGES) - 1) & 1u, p.timeout_ns))
        return false;
      if (__any_sync(kFull, *(volatile int *)&abort_flag)) return false;
      if (lane == 0) mbar_arrive_expect_tx(&v_full[vs], Cfg::KV_BYTES);
      __syncwarp();
      if (lane < Cfg::LOADS)
        tma_load_2d(sV + (size_t)vs * Cfg::KV_BYTES + panel * Cfg::PANEL_KV + slot * 2048, &tmV, panel * 64,
                    (int)(trow * kBlock), &v_full[vs]);
      if (lane == 0) v_issued = g + 1;
      return true;
    };
    const bool vw = warp == Cfg::V_PRODUCER;
    bool ok = true;
    const Pend nil{0, 0, true};
    bool h0 = step();  // tiles g, g + 1, g + 2 exist (the cursor one further on)
    Pend f0 = h0 ? fetch() : nil;
    bool h1 = h0 && step();
    Pend f1 = h1 ? fetch() : nil;
    bool h2 = h1 && step();
    Pend f2 = h2 ? fetch() : nil;
    for (int g = 0; h0 && ok; ++g) {
      const bool h3 = h2 && step();
      const Pend f3 = h3 ? fetch() : nil;
      const int64_t r = row_of(f0);
      ok = vw ? issue_v(g, r) : issue_k(g, r);
      h0 = h1;
      f0 = f1;
      h1 = h2;
      f1 = f2;
      h2 = h3;
      f2 = f3;
    }
    if (__any_sync(kFull, bad)) {
      if (lane == 0) atomicOr(&cta_flags, PKV_FLAG_BAD_BLOCK);
    }
    if (!ok && lane == 0) {
      atomicOr(&cta_flags, PKV_FLAG_TIMEOUT);
      abort_flag = 1;
    }
  } else if (warp == Cfg::ISSUER) {
    // ---------------- S issue (P . V has a warp of its own) ----------------
    const uint32_t q0 = smem_u32(sQ);
    bool ok = true;
    int g = 0;      // global K / V tile
    int items = 0;  // valid items so far (Q phases)
    // S = Q . K^T of global tile gg into S buffer gg % SBUF (free once P . V of
    // tile gg - SBUF, which read P from it, is done)
    auto issue_s = [&](int gg) -> bool {
      const int ks = gg % Cfg::KSTAGES, sb = gg % Cfg::SBUF;
      if (!warp_wait(&k_full[ks], (uint32_t)(gg / Cfg::KSTAGES) & 1u, p.timeout_ns)) return false;
      if (gg >= Cfg::SBUF && !warp_wait(&pv_done[sb], (uint32_t)((gg / Cfg::SBUF) - 1) & 1u, p.timeout_ns))
        return false;
      if (lane == 0) k_consumed = gg + 1;
      tc::fence_after();
      if (lane == 0) {
        mma_s_tile<Cfg>(tbase + (uint32_t)(sb * Cfg::N), q0, smem_u32(sK + (size_t)ks * Cfg::KV_BYTES));
        tc::commit(&s_full[sb]);
        tc::commit(&k_empty[ks]);
      }
      __syncwarp();
      return true;
    };
    for (int k = 0; k < n_rounds && ok; ++k) {
      const int i = round_item(k);
      if (i >= n_items) continue;
      const PrefillItem it = prefill_item<Cfg>(p, i);
      if (!it.valid || it.T == 0) continue;
      // this item's Q is staged (only items with tiles stage one)
      ok = warp_wait(&q_full, (uint32_t)items & 1u, p.timeout_ns);
      ++items;
      if (!ok) break;
      tc::fence_after();
      for (int j = 0; j < it.T && ok; ++j) {
        ok = issue_s(g + j);
        if (ok && __any_sync(kFull, *(volatile int *)&abort_flag)) ok = false;
      }
      g += it.T;
    }
    if (!ok && lane == 0) {
      atomicOr(&cta_flags, PKV_FLAG_TIMEOUT);
      abort_flag = 1;
    }
  } else if (warp == Cfg::PV_ISSUER) {
    // ---------------- P . V issue ----------------
    bool ok = true;
    int g = 0;        // global K / V tile
    int o_items = 0;  // items with tiles so far (O hand-offs)
    for (int k = 0; k < n_rounds && ok; ++k) {
      const int i = round_item(k);
      if (i >= n_items) continue;
      const PrefillItem it = prefill_item<Cfg>(p, i);
      if (!it.valid || it.T == 0) continue;
      for (int j = 0; j < it.T && ok; ++j) {
        const int gj = g + j;
        const int vs = gj % Cfg::VSTAGES, sb = gj % Cfg::SBUF;
        // the first P . V of an item overwrites O: the previous item's O must be read out
        if (j == 0 && o_items > 0 && !(ok = warp_wait(&o_free, (uint32_t)(o_items - 1) & 1u, p.timeout_ns))) break;
        ok = warp_wait(&v_full[vs], (uint32_t)(gj / Cfg::VSTAGES) & 1u, p.timeout_ns);
        if (ok) ok = warp_wait(&p_full[sb], (uint32_t)(gj / Cfg::SBUF) & 1u, p.timeout_ns);
        if (!ok) break;
        if (lane == 0) v_consumed = gj + 1;
        uint8_t *vt = sV + (size_t)vs * Cfg::KV_BYTES;
        {  // stale cache rows past the context: weight 0, but 0 * NaN is NaN
          const int kv0 = (it.j_first + j) * Cfg::N;  // first position of the tile
          zero_v_rows<Cfg>(vt, it.ctx - kv0, min(it.nblk * kBlock - kv0, Cfg::N), lane);
        }
        __syncwarp();
        tc::fence_after();
        if (lane == 0) {
          mma_pv_tile<Cfg>(tbase + Cfg::COL_O, tbase + (uint32_t)(sb * Cfg::N), smem_u32(vt), j > 0);
          tc::commit(&pv_done[sb]);
          tc::commit(&v_empty[vs]);
        }
        __syncwarp();
        if (__any_sync(kFull, *(volatile int *)&abort_flag)) ok = false;
      }
      g += it.T;
      ++o_items;
    }
    if (!ok && lane == 0) {
      atomicOr(&cta_flags, PKV_FLAG_TIMEOUT);
      abort_flag = 1;
    }
  } else {
    // ---------------- softmax + epilogue: thread (row, half) ----------------
    constexpr int SC = Cfg::N / 2;  // S columns of a thread (its half of the row)
    constexpr int OC = Cfg::D / 2;  // O columns of a thread
    const int row = tid & (Cfg::M - 1), half = tid / Cfg::M;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const float c = p.scale_log2;
    // where thread (row, half) reads row `row` of item i's Q tile (null past R: zeros)
    auto q_src = [&](int i) -> const uint4 * {
      const PrefillItem it = prefill_item<Cfg>(p, i);
      const int r = it.r0 + row;
      const int ii = r / p.G, g = r - ii * p.G;
      return r < it.R ? reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(p.q) +
                                                       ((size_t)(it.qs + ii) * p.Hq + it.h * p.G + g) * Cfg::D)
                      : nullptr;
    };
    // thread (row, half) stages its half of a Q row from `src`
    auto stage_q = [&](const uint4 *src, bool async) {
#pragma unroll
      for (int k = 0; k < Cfg::D / 16; ++k) {
        const int cc = half * (Cfg::D / 16) + k;
        const uint32_t dst = smem_u32(sQ + (cc >> 3) * Cfg::PANEL_Q + row * 128 + (((cc & 7) ^ (row & 7)) << 4));
        if (src && async)
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src + cc) : "memory");
        else
          sts128(dst, src ? __ldg(src + cc) : make_uint4(0, 0, 0, 0));
      }
    };
    auto release_q = [&](bool async) {
      if (async) asm volatile("cp.async.wait_all;" ::: "memory");
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(&q_full);
    };
    // Q is staged for the CTA's items with tiles only, one after another: Q of
    // the next such item is released after this one's last S has landed, so
    // the MMA warp has waited for every earlier Q (no barrier phase is skipped)
    auto next_work = [&](int k) {  // the first round from k on whose item has tiles (or n_rounds)
      for (; k < n_rounds; ++k) {
        const int i = round_item(k);
        if (i >= n_items) continue;
        const PrefillItem t = prefill_item<Cfg>(p, i);
        if (t.valid && t.T > 0) break;
      }
      return k;
    };
    // Lookahead: `kn2` is the round of the item with tiles after the one whose
    // Q is staged, and `src2` where this thread reads that item's Q row.  Both
    // are looked up while an epilogue waits for its item's last P . V, so the
    // last tile of an item (which stages the next Q) does no global loads.
    int kn2 = n_rounds;
    const uint4 *src2 = nullptr;
    {
      const int first = next_work(0);
      if (first < n_rounds) {
        stage_q(q_src(round_item(first)), false);
        release_q(false);
        kn2 = next_work(first + 1);
        if (kn2 < n_rounds) src2 = q_src(round_item(kn2));
      }
    }
    bool ok = true;
    int g = 0;        // global tile (S buffers, exchange parity)
    int o_items = 0;  // items with tiles so far
    for (int k = 0; k < n_rounds && ok; ++k) {
      const int cur = round_item(k);
      if (cur >= n_items) continue;
      const PrefillItem it = prefill_item<Cfg>(p, cur);
      if (tid == 0 && (it.bad_q || it.bad_ctx)) atomicOr(&cta_flags, PKV_FLAG_BAD_LEN);
      if (!it.valid) continue;
      const int T = it.T, j_first = it.j_first;
      const int r = it.r0 + row;
      const bool valid = r < it.R;
      const int lim = valid ? it.ctx - it.n + r / p.G + 1 : 0;  // visible positions [lo, lim)
      const int lo = (valid && p.window > 0) ? max(0, lim - p.window) : 0;
      const int ii = r / p.G, gq = r - ii * p.G;
      uint4 *dst = valid ? reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.out) +
                                                     ((size_t)(it.qs + ii) * p.Hq + it.h * p.G + gq) * Cfg::D +
                                                     half * OC)
                         : nullptr;
      float m_run = -INFINITY, l = 0.f;
      bool staged = false;  // the next item's Q copy is in flight
      for (int j = 0; j < T; ++j) {
        const int gj = g + j, sb = gj % Cfg::SBUF;
        // failure-path test hook: the first tile's wait is on a barrier
        // nothing completes, so it runs out and the CTA takes its abort path
        ok = (p.stall_ns != 0 && gj == 0)
                 ? warp_wait(&dead, 0, p.timeout_ns)
                 : warp_wait(&s_full[sb], (uint32_t)(gj / Cfg::SBUF) & 1u, p.timeout_ns);
        if (!ok) break;
        tc::fence_after();
        const uint32_t scol = tbase + lane_base + (uint32_t)(sb * Cfg::N + half * SC);
        uint32_t s[SC / 32][32];
#pragma unroll
        for (int q = 0; q < SC / 32; ++q) tc::ld32(scol + (uint32_t)(q * 32), s[q]);
        if (j + 1 == T) {
          // every S MMA of this item has completed (its last S just landed):
          // the next item's Q can replace this one's while the softmax runs
          if (kn2 < n_rounds) {
            stage_q(src2, true);
            staged = true;
          }
        }
        const int kv0 = (j_first + j) * Cfg::N + half * SC;
        if (!(kv0 >= lo && kv0 + SC <= lim)) {  // a mask edge crosses these columns
#pragma unroll
          for (int q = 0; q < SC / 32; ++q)
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const int pos = kv0 + q * 32 + e;
              if (pos < lo || pos >= lim) s[q][e] = 0xff800000u;  // -inf
            }
        }
        float mx = -INFINITY;
#pragma unroll
        for (int q = 0; q < SC / 32; ++q)
#pragma unroll
          for (int e = 0; e < 32; e += 2) mx = fmax3(mx, __uint_as_float(s[q][e]), __uint_as_float(s[q][e + 1]));
        // the row max over both halves (double-buffered exchange, bounded wait)
        red[gj & 1][half][row] = mx;
        __syncwarp();
        if (lane == 0) mbar_arrive(&xch[warp & 3][gj & 1]);
        ok = warp_wait(&xch[warp & 3][gj & 1], (uint32_t)(gj >> 1) & 1u, p.timeout_ns);
        if (!ok) break;
        mx = fmaxf(mx, red[gj & 1][half ^ 1][row]);
        const float m_new = fmaxf(m_run, mx * c);
        // warps w and w + 4 hold the same rows and the same m_new: same decision
        const bool rescale = __any_sync(kFull, m_new > m_run + 8.f);
        float alpha = 1.f;
        if (rescale) {
          alpha = m_new == -INFINITY ? 1.f : ex2(m_run - m_new);
          m_run = m_new;
        }
        const float mu = m_run == -INFINITY ? 0.f : m_run;
        const uint64_t cmu = f2_pack(c, c), nmu = f2_pack(-mu, -mu);
        uint64_t sum2 = f2_pack(0.f, 0.f);
        uint32_t w[SC / 2], wl[Cfg::BF ? SC / 2 : 1];
#pragma unroll
        for (int e = 0; e < SC / 2; ++e) {
          const int col = 2 * e;
          uint32_t lo_;
          p_pair<Cfg::BF>(s[col >> 5][col & 31], s[(col + 1) >> 5][(col + 1) & 31], cmu, nmu, sum2, w[e], lo_);
          if constexpr (Cfg::BF) wl[e] = lo_;
        }
        const float2 sp = f2_unpack(sum2);
        const float sum = sp.x + sp.y;
        l = l * alpha + sum;
        // P over this thread's own (already read) S columns
        tc::st32(scol, w);
        if constexpr (Cfg::BF) tc::st32(scol + 32, wl);
        // O must hold P . V of the previous tile before it is scaled, and be
        // scaled before P . V of this tile (issued after the arrival below)
        if (rescale && j > 0) {
          ok = warp_wait(&pv_done[(gj - 1) % Cfg::SBUF], (uint32_t)((gj - 1) / Cfg::SBUF) & 1u, p.timeout_ns);
          if (!ok) break;
          tc::fence_after();
          scale_o<Cfg>(tbase + lane_base + Cfg::COL_O + (uint32_t)(half * OC), alpha);
        }
        tc::wait_st();
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[sb]);
      }
      if (!ok) break;
      // the next item's Q: its copy overlapped this item's last tile
      if (staged) {
        release_q(true);
        kn2 = next_work(kn2 + 1);  // and the item after it, while the last P . V runs
        src2 = kn2 < n_rounds ? q_src(round_item(kn2)) : nullptr;
      }
      // epilogue: O of this item
      if (T > 0) {
        const int gl = g + T - 1;
        ok = warp_wait(&pv_done[gl % Cfg::SBUF], (uint32_t)(gl / Cfg::SBUF) & 1u, p.timeout_ns);
        if (ok) {  // the row sum over both halves
          red_l[half][row] = l;
          __syncwarp();
          if (lane == 0) mbar_arrive(&xl[warp & 3]);
          ok = warp_wait(&xl[warp & 3], (uint32_t)o_items & 1u, p.timeout_ns);
        }
        if (!ok) break;
        tc::fence_after();
        const float lt = l + red_l[half ^ 1][row];
        const float inv = lt > 0.f ? 1.f / lt : 0.f;  // a row that sees nothing gives 0
        uint32_t o[OC / 32][32];
#pragma unroll
        for (int q = 0; q < OC / 32; ++q) tc::ld32(tbase + lane_base + Cfg::COL_O + (uint32_t)(half * OC + q * 32), o[q]);
        // O is in registers: the next item's P . V may overwrite it, and the
        // row sums may be overwritten by the next exchange
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&o_free);
        store_rows_staged<Cfg>(o, inv, dst, sO + (size_t)(warp * 2048), lane);
        ++o_items;
      } else if (dst) {  // no visible position for any row of the tile: zeros
#pragma unroll
        for (int q = 0; q < OC / 8; ++q) dst[q] = make_uint4(0, 0, 0, 0);
      }
      g += T;
    }
    if (!ok && lane == 0) {
      atomicOr(&cta_flags, PKV_FLAG_TIMEOUT);
      abort_flag = 1;
    }
  }

  // ---------------- drain, then free tensor memory ----------------
  tc::fence_before();
  __syncthreads();
  if (warp == Cfg::ISSUER || warp == Cfg::PV_ISSUER) {
    if (lane == 0) tc::commit(&fin);  // completes once every MMA either warp issued has
    __syncwarp();
    if (!mbar_wait_bounded(&fin, 0, p.timeout_ns) && lane == 0) atomicOr(&cta_flags, PKV_FLAG_TIMEOUT);
  } else if (warp == Cfg::PRODUCER && lane == 0) {  // copies issued but never consumed (abort only)
    for (int j = k_consumed; j < k_issued; ++j)
      mbar_wait_bounded(&k_full[j % Cfg::KSTAGES], (uint32_t)(j / Cfg::KSTAGES) & 1u, p.timeout_ns);
    for (int j = v_consumed; j < v_issued; ++j)
      mbar_wait_bounded(&v_full[j % Cfg::VSTAGES], (uint32_t)(j / Cfg::VSTAGES) & 1u, p.timeout_ns);
  } else if (tid < Cfg::SOFTMAX) {
    asm volatile("cp.async.wait_all;" ::: "memory");  // a Q copy left in flight by an abort
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == Cfg::ISSUER) tc::dealloc(tbase, Cfg::TMEM_COLS);
  if (tid == 0 && cta_flags && p.status) atomicOr(p.status, cta_flags);
}

template <class Cfg>
static cudaError_t launch_cfg(const PrefillParams &p, const CUtensorMap &tmK, const CUtensorMap &tmV,
                              cudaStream_t stream) {
  static int configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorNotSupported;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(prefill_kernel<Cfg>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)(Cfg::SMEM + kOutStage));
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  static int sms[64] = {};
  if (!sms[dev]) {
    e = cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
  }
  const int64_t items = (int64_t)p.max_tiles * p.Hkv * p.B;
  if (items > INT32_MAX) return cudaErrorInvalidValue;
  const unsigned grid = (unsigned)(items < sms[dev] ? items : sms[dev]);  // one persistent CTA per SM
  static_assert(Cfg::SMEM + kOutStage + 4096 <= 232448, "shared memory");
  prefill_kernel<Cfg><<<grid, Cfg::THREADS, Cfg::SMEM + kOutStage, stream>>>(p, tmK, tmV);
  return cudaGetLastError();
}

cudaError_t launch_prefill(const PrefillParams &p, int cache_dtype, const CUtensorMap &tmK, const CUtensorMap &tmV,
                           cudaStream_t stream) {
  if (p.max_tiles <= 0 || p.B <= 0) return cudaSuccess;
  if (cache_dtype == PKV_BF16) {
    if (p.D == 128) return launch_cfg<PrefillCfg<BF16, 128>>(p, tmK, tmV, stream);
    if (p.D == 64) return launch_cfg<PrefillCfg<BF16, 64>>(p, tmK, tmV, stream);
  } else if (cache_dtype == PKV_F16) {
    if (p.D == 128) return launch_cfg<PrefillCfg<F16, 128>>(p, tmK, tmV, stream);
    if (p.D == 64) return launch_cfg<PrefillCfg<F16, 64>>(p, tmK, tmV, stream);
  }
  return cudaErrorNotSupported;
}

}  // namespace pkv
