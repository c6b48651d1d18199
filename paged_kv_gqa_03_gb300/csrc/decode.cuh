// decode.cuh — the paged decode-attention kernel (steps a4–a8 up to the
// partial results), templated on cache dtype, head dim and compute path.
//
// Work decomposition.  A "unit" is (sequence b, kv head h, row chunk c): the
// query rows c*GC ... (at most GC of them) of the R = q_len * G rows that
// share kv head h ("大模型推理加速——KV Cache篇" §6.2 GQA).  Row r is query head
// h*G + r % G of new token r / G; with q_len > 1 (several new tokens per
// sequence, the verify step of speculative decoding, "LLM推理优化实战" §4) new
// token i sees only the first ctx - (q_len - 1 - i) positions, the causal mask
// tril(diagonal = kv_len - q_len) of "苦猿的大模型日记 Day45" PART 04, applied
// per score column.  With a sliding window W (the same page, PART 02: a fixed
// visible history) a row sees only [lim - W, lim); a unit then streams only
// the blocks from the first one row 0's window reaches.  Units are
// concatenated in the order
// (b, h, c), each contributing ceil(ctx_b / 16) block items, and the item list
// is cut into P equal contiguous ranges, one per warp (the "workers").  A
// warp streams its range block by block, carrying the online-softmax state
// across blocks of a unit ("LLM推理优化实战" §3.2 online softmax: running max
// m, running sum l, accumulator rescaled by exp(m_old - m_new)); a unit cut by
// a range boundary leaves normalised (o, lse) partials that the merge kernel
// combines (log-sum-exp rule).  (Letting the last warp of each split unit merge
// it inside this kernel measured ~2 % slower on GB300: a unit's last partial
// always lands at the end of some warp's range, so the fused merge only moved
// serial work into the kernel's tail.)
//
// Data movement.  Each warp owns a ring of STAGES shared-memory slots; lane 0
// issues 2-D TMA loads (cp.async.bulk.tensor, 128-byte swizzle) of the block's
// K tile and V tile — each a contiguous 16 x D run of [num_blocks][Hkv][16][D]
// reached through the block table ("LLM推理优化实战" §2.2 block table) — onto
// the slot's mbarrier, STAGES blocks ahead of the consumer.
//
// Compute.  MMA path (f16/bf16/fp8 caches): per 16-token block,
// S^T[16 tok x 8 rows] = K[16 x D] . Q^T[D x 8] and O^T[D x 8] += V^T[D x 16] .
// P^T[16 x 8] with mma.sync m16n8k16 (fp32 accumulate); P moves from the
// score fragment to the B operand with movmatrix.  Units serve 8 rows; on
// fp8 caches a kv head with more than 8 rows (several new tokens per
// sequence) is served in 16-row units, two 8-row column groups per MMA A
// operand, so each E4M3 K / V element is widened to f16 once per 16 rows.  CUDA-core path (fp32
// caches, groups of 1-2): lanes split tokens for q.K and head-dim slices for
// p.V.  Scores use the scale of "苦猿的大模型日记 Day45" PART 02
// (softmax(QK^T / sqrt(d))), applied in fp32 in the log2 domain.
#pragma once

#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace pkv {

// BPS_ = blocks per pipeline stage.  2 (fp8 tensor-core path only): a stage
// holds two consecutive blocks of one unit, which share one barrier, one
// stage record, one online-softmax update (one max exchange, one accumulator
// rescale per 32 tokens) and one producer step — an fp8 block carries half a
// 16-bit block's bytes for the same per-block instructions, which made the
// one-block fp8 kernel issue-bound.
template <class CacheT, class QT, int D_, int GC_, bool MMA_, int WARPS_, int BUDGET_, int BPS_ = 1>
struct DecodeCfg {
  using Cache = CacheT;
  using Q = QT;
  static constexpr int D = D_, GC = GC_, WARPS = WARPS_, BPS = BPS_;
  static constexpr bool MMA = MMA_;
  static constexpr bool FP8 = CacheT::kBytes == 1;
  static constexpr int ROWB = D * CacheT::kBytes;           // bytes per token row
  static constexpr int TILE = kBlock * ROWB;                // bytes per (block, head) tile
  static constexpr int STAGE_BYTES = BPS * 2 * TILE;        // K and V tiles of a stage's blocks
  static constexpr int STAGES_RAW = BUDGET_ / STAGE_BYTES;
  static constexpr int STAGES = STAGES_RAW < 2 ? 2 : (STAGES_RAW > 8 ? 8 : STAGES_RAW);
  static constexpr int NBOX = ROWB >= 128 ? ROWB / 128 : 1;  // TMA boxes per tile
  static constexpr int BOX_ROWS = ROWB >= 128 ? kBlock : kBlock * ROWB / 128;
  static constexpr int BOX_ELEMS = 128 / CacheT::kBytes;
  static constexpr size_t TILES_BYTES = (size_t)WARPS * STAGES * STAGE_BYTES;
  static constexpr size_t META_BYTES = (size_t)WARPS * STAGES * sizeof(StageMeta);
  static constexpr size_t BAR_BYTES = (size_t)WARPS * STAGES * 8;
  static constexpr size_t QBUF_BYTES = MMA ? 0 : (size_t)WARPS * GC * D * 4;
  static constexpr size_t PREFIX_BYTES = (size_t)kInlinePrefix * 4;  // inline plan
  static constexpr size_t SMEM = 1024 + TILES_BYTES + META_BYTES + BAR_BYTES + QBUF_BYTES + PREFIX_BYTES;
  // CTAs that fit in an SM's 228 KiB of shared memory (1 KiB reserved per CTA);
  // passed to __launch_bounds__ so registers never limit residency further
  static constexpr int CTAS_RAW = (int)(233472 / (SMEM + 1024));
  static constexpr int MIN_CTAS = CTAS_RAW < 1 ? 1 : (CTAS_RAW > 8 ? 8 : CTAS_RAW);
  static_assert(TILE % 1024 == 0, "tiles must keep 1024-byte alignment for the swizzle");
  static_assert(!MMA || GC == 8 || (GC == 16 && FP8 && BPS == 2),
                "the MMA path serves 8-row units (16-row units: the two-block fp8 path)");
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(BPS == 1 || (BPS == 2 && MMA && FP8), "two blocks per stage: the fp8 tensor-core path");
};

// ---------------------------------------------------------------------------
// Producer: walks the worker's item range and issues TMA loads.
// ---------------------------------------------------------------------------
struct Producer {
  int pi, e, s;          // next item, end of range, start of range
  int b, hu, j, n, ctx;  // unit and block of item pi; blocks and length of sequence b
  int j0;                // first block of sequence b inside some row's window
  int seg_j0, seg_wfirst;
  int win_b, win_hu, win_j0, win_id;  // lane-parallel window of 32 block-table entries
  int nxt_id;                         // the unit's next window, loaded one window ahead
  float win_ks, win_vs;
};

__device__ __forceinline__ void load_seq(Producer &pr, const DecodeParams &p) {
  const int ctx = clamped_len(p, __ldg(p.context_lens + pr.b));
  pr.ctx = ctx;
  pr.n = (ctx + kBlock - 1) / kBlock;
  pr.j0 = first_block(p, ctx);
}

// Block-table entry (and, for fp8, the block's K / V scales) of block jj of
// the producer's current unit, from the lane-parallel window of 32 entries;
// the window moves to start at jj when jj leaves it (the following window
// is loaded one window ahead).
template <class Cfg>
__device__ __forceinline__ int window_block(Producer &pr, const DecodeParams &p, int jj, int h, int lane,
                                            float &ks, float &vs) {
  if (!(pr.b == pr.win_b && pr.hu == pr.win_hu && jj >= pr.win_j0 && jj < pr.win_j0 + 32)) {
    const int32_t *row = p.block_table + (size_t)pr.b * p.max_blocks;
    if (pr.b == pr.win_b && pr.hu == pr.win_hu && jj == pr.win_j0 + 32) {
      pr.win_id = pr.nxt_id;  // the window loaded ahead
    } else {
      const int jw = jj + lane;
      pr.win_id = jw < pr.n ? __ldg(row + jw) : 0;
    }
    pr.win_b = pr.b;
    pr.win_hu = pr.hu;
    pr.win_j0 = jj;
    // load the following window now; it is first needed 32 blocks later
    const int jn = jj + 32 + lane;
    pr.nxt_id = jn < pr.n ? __ldg(row + jn) : 0;
    if constexpr (Cfg::FP8) {
      const int jw = jj + lane, id = pr.win_id;
      float a = 0.f, c = 0.f;
      if (jw < pr.n && id >= 0 && (int64_t)id < p.num_blocks) {
        a = __ldg(p.k_scale + (size_t)id * p.Hkv + h);
        c = __ldg(p.v_scale + (size_t)id * p.Hkv + h);
      }
      pr.win_ks = a;
      pr.win_vs = c;
    }
  }
  const int blk = __shfl_sync(kFull, pr.win_id, jj - pr.win_j0);
  ks = vs = 1.f;
  if constexpr (Cfg::FP8) {
    ks = __shfl_sync(kFull, pr.win_ks, jj - pr.win_j0);
    vs = __shfl_sync(kFull, pr.win_vs, jj - pr.win_j0);
  }
  return blk;
}

// Lane 0: the TMA copies of one block's K and V tiles to dk / dv, onto bar.
// A bad id reads the tile just past the end of the tensor: TMA fills zeros.
template <class Cfg>
__device__ __forceinline__ void issue_block(const DecodeParams &p, const CUtensorMap *tmK, const CUtensorMap *tmV,
                                            uint8_t *dk, uint8_t *dv, int blk, int h, uint64_t *bar,
                                            int *cta_flags) {
  const bool bad = blk < 0 || (int64_t)blk >= p.num_blocks;
  const int64_t tile_row = bad ? p.num_blocks * p.Hkv : (int64_t)blk * p.Hkv + h;
  if (bad) atomicOr(cta_flags, PKV_FLAG_BAD_BLOCK);
  const int y = (int)(tile_row * Cfg::BOX_ROWS);
#pragma unroll
  for (int bx = 0; bx < Cfg::NBOX; ++bx) {
    tma_load_2d(dk + bx * 2048, tmK, bx * Cfg::BOX_ELEMS, y, bar);
    tma_load_2d(dv + bx * 2048, tmV, bx * Cfg::BOX_ELEMS, y, bar);
  }
}

// Fills pipeline stage `stage` with the worker's next item (with BPS = 2 also
// the one after it, when it is the next block of the same unit and inside the
// worker's range) and advances the producer; returns the blocks issued.
template <class Cfg>
__device__ __forceinline__ int produce(Producer &pr, const DecodeParams &p, const CUtensorMap *tmK,
                                       const CUtensorMap *tmV, uint8_t *tiles, StageMeta *meta,
                                       uint64_t *bars, int stage, int lane, int *cta_flags) {
  __syncwarp();
  const int h = pr.hu / p.NC;
  float ks, vs, ks1 = 1.f, vs1 = 1.f;
  const int blk = window_block<Cfg>(pr, p, pr.j, h, lane, ks, vs);
  int nb = 1, blk1 = 0;
  if constexpr (Cfg::BPS == 2) {
    if (pr.pi + 1 < pr.e && pr.j + 1 < pr.n) {
      nb = 2;
      blk1 = window_block<Cfg>(pr, p, pr.j + 1, h, lane, ks1, vs1);
    }
  }
  int flags = 0;
  if (pr.pi == pr.s || pr.j == pr.j0) {
    flags |= kFirst;
    pr.seg_j0 = pr.j;
    pr.seg_wfirst = (pr.pi == pr.s);
  }
  const int jl = pr.j + nb - 1;  // the stage's last block
  if (pr.pi + nb == pr.e || jl + 1 == pr.n) {
    flags |= kLast;
    if (pr.seg_j0 == pr.j0 && jl + 1 == pr.n) flags |= kComplete;
  }
  if (pr.seg_wfirst) flags |= kWFirst;
  const int rem = pr.ctx - pr.j * kBlock;
  const int nvalid = min(kBlock, rem);
  if (lane == 0) {
    StageMeta m;
    m.b = pr.b;
    m.hu = pr.hu;
    m.j = pr.j;
    m.nvalid = nvalid;
    m.ks = ks;
    m.vs = vs;
    m.flags = flags;
    m.rem = rem;
    m.ks1 = ks1;
    m.vs1 = vs1;
    m.nb = nb;
    m.pad = 0;
    meta[stage] = m;
    // the warp's reads of this stage have completed (their results were
    // consumed), so the TMA overwrite needs no proxy fence here
    mbar_arrive_expect_tx(&bars[stage], nb * 2 * Cfg::TILE);
    uint8_t *dk = tiles + (size_t)stage * Cfg::STAGE_BYTES;
    issue_block<Cfg>(p, tmK, tmV, dk, dk + Cfg::TILE, blk, h, &bars[stage], cta_flags);
    if (nb == 2) issue_block<Cfg>(p, tmK, tmV, dk + 2 * Cfg::TILE, dk + 3 * Cfg::TILE, blk1, h, &bars[stage], cta_flags);
  }
  // advance past the stage's items
  pr.pi += nb;
  pr.j += nb;
  if (pr.j == pr.n && pr.pi < pr.e) {
    if (++pr.hu == p.HU) {
      pr.hu = 0;
      do {
        ++pr.b;
        load_seq(pr, p);
      } while (pr.n == 0 && pr.b < p.B - 1);
    }
    pr.j = pr.j0;
  }
  return nb;
}

// Zeroes token rows [nvalid, 16) of a tile so stale (possibly non-finite)
// cache contents cannot leak into p.V through a zero weight.
template <int ROWB>
__device__ __forceinline__ void zero_tail_rows(uint8_t *tile, int nvalid, int lane) {
  constexpr int CPR = ROWB / 16;  // 16-byte chunks per row
  const uint32_t base = smem_u32(tile);
  for (int idx = lane; idx < (kBlock - nvalid) * CPR; idx += 32) {
    const int row = nvalid + idx / CPR, ch = idx % CPR;
    sts128(base + tile_off<ROWB>(row, ch * 16), make_uint4(0, 0, 0, 0));
  }
  fence_proxy_async();
  __syncwarp();
}

// Row r (0 <= r < R) of kv head h of sequence b: its offset in q / out,
// [B][q_len][Hq][D] (q_len = 1: [B][Hq][D]), in elements.
__device__ __forceinline__ size_t query_row(const DecodeParams &p, int b, int h, int r) {
  const int i = r / p.G;
  return (((size_t)b * p.q_len + i) * p.Hq + h * p.G + (r - i * p.G)) * (size_t)p.D;
}

// Positions hidden from row r at the end of the sequence: the newer tokens of
// its step, q_len - 1 - r / G (0 for rows past R, which are padding).
__device__ __forceinline__ int row_back(const DecodeParams &p, int r) {
  return max(0, p.q_len - 1 - r / p.G);
}

// ---------------------------------------------------------------------------
// MMA path state and steps.
// ---------------------------------------------------------------------------
template <class Cfg>
struct MmaState {
  static constexpr int KS = Cfg::D / 16;  // k-steps of q.K
  static constexpr int MT = Cfg::D / 16;  // m-tiles of V^T
  static constexpr int NH = Cfg::GC >= 8 ? Cfg::GC / 8 : 1;  // 8-row column groups of a unit
  uint32_t qb[NH][KS][2];
  float acc[NH][MT][4];
  float m[NH][2], l[NH][2];  // per score column 8 nh + 2 tig, 8 nh + 2 tig + 1
  int back[NH][2];           // row_back of those columns
  int bk_lo, bk_hi;          // least and largest row_back over the unit's rows
};

template <class Cfg>
__device__ __forceinline__ void mma_begin(MmaState<Cfg> &st, const DecodeParams &p, const StageMeta &m,
                                          int lane) {
  const int gid = lane >> 2, tig = lane & 3;
  const int h = m.hu / p.NC, r0 = (m.hu % p.NC) * Cfg::GC;
  const int gc = min(Cfg::GC, p.R - r0);
  st.bk_lo = row_back(p, r0 + Cfg::GC - 1);  // row_back does not grow with the row
  st.bk_hi = row_back(p, r0);
#pragma unroll
  for (int nh = 0; nh < MmaState<Cfg>::NH; ++nh) {
    const int rq = 8 * nh + gid;  // the q row (B-operand column) this lane loads
    const size_t row = rq < gc ? query_row(p, m.b, h, r0 + rq) : 0;
    st.back[nh][0] = row_back(p, r0 + 8 * nh + 2 * tig);
    st.back[nh][1] = row_back(p, r0 + 8 * nh + 2 * tig + 1);
#pragma unroll
    for (int ks = 0; ks < MmaState<Cfg>::KS; ++ks) {
      uint32_t b0 = 0, b1 = 0;
      if (rq < gc) {
        if constexpr (Cfg::FP8) {
          // k-slots 2t,2t+1 | 2t+8,2t+9 hold d = 16ks + 4t + {0,1} | {2,3}
          const uint2 raw = *reinterpret_cast<const uint2 *>(
              reinterpret_cast<const uint16_t *>(p.q) + row + 16 * ks + 4 * tig);
          float2 x0, x1;
          if constexpr (Cfg::Q::kCode == PKV_BF16) {
            x0 = unpack2(BF16{}, raw.x);
            x1 = unpack2(BF16{}, raw.y);
          } else {
            x0 = unpack2(F16{}, raw.x);
            x1 = unpack2(F16{}, raw.y);
          }
          b0 = pack_f16x2(x0.x, x0.y);
          b1 = pack_f16x2(x1.x, x1.y);
        } else {
          const uint16_t *qr = reinterpret_cast<const uint16_t *>(p.q) + row + 16 * ks + 2 * tig;
          b0 = *reinterpret_cast<const uint32_t *>(qr);
          b1 = *reinterpret_cast<const uint32_t *>(qr + 8);
        }
      }
      st.qb[nh][ks][0] = b0;
      st.qb[nh][ks][1] = b1;
    }
#pragma unroll
    for (int mt = 0; mt < MmaState<Cfg>::MT; ++mt)
#pragma unroll
      for (int r = 0; r < 4; ++r) st.acc[nh][mt][r] = 0.f;
    st.m[nh][0] = st.m[nh][1] = -INFINITY;
    st.l[nh][0] = st.l[nh][1] = 0.f;
  }
}

// A block's K and V operands in registers (MMA fragments, or raw fp8 words).
template <class Cfg>
struct MmaFrags {
  static constexpr int KS = Cfg::D / 16, MT = Cfg::D / 16;
  static constexpr int KW = Cfg::FP8 ? 2 : 4;            // words per k-step
  static constexpr int VW = Cfg::FP8 ? Cfg::D / 32 : 4;  // words per token row (fp8) / m-tile
  static constexpr int VN = Cfg::FP8 ? 4 : MT;           // fp8: 4 token rows
  uint32_t k[KS][KW];
  uint32_t v[VN][VW];
};

template <class Cfg>
__device__ __forceinline__ void mma_load(MmaFrags<Cfg> &f, uint8_t *tk, uint8_t *tv, int nvalid, int lane) {
  constexpr int ROWB = Cfg::ROWB;
  const int gid = lane >> 2, tig = lane & 3;
  const uint32_t kb = smem_u32(tk), vb = smem_u32(tv);
  if (nvalid < kBlock) zero_tail_rows<ROWB>(tv, nvalid, lane);
  if constexpr (Cfg::FP8) {
#pragma unroll
    for (int ks = 0; ks < MmaFrags<Cfg>::KS; ++ks) {
      f.k[ks][0] = lds32(kb + tile_off<ROWB>(gid, 16 * ks + 4 * tig));
      f.k[ks][1] = lds32(kb + tile_off<ROWB>(gid + 8, 16 * ks + 4 * tig));
    }
    constexpr int DPT = Cfg::D / 8;  // head-dim bytes owned by one row group
    const int trow[4] = {2 * tig, 2 * tig + 1, 2 * tig + 8, 2 * tig + 9};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if constexpr (DPT == 16) {
        const uint4 r = lds128(vb + tile_off<ROWB>(trow[i], 16 * gid));
        f.v[i][0] = r.x; f.v[i][1] = r.y; f.v[i][2] = r.z; f.v[i][3] = r.w;
      } else {
        const uint2 r = lds64(vb + tile_off<ROWB>(trow[i], 8 * gid));
        f.v[i][0] = r.x; f.v[i][1] = r.y;
      }
    }
  } else {
    const int r = lane & 7, mi = lane >> 3;
    const int krow = r + ((mi & 1) << 3), khi = mi >> 1;
    const int vtok = r + ((mi >> 1) << 3), vhi = mi & 1;
#pragma unroll
    for (int ks = 0; ks < MmaFrags<Cfg>::KS; ++ks) ldsm_x4(kb + tile_off<ROWB>(krow, (2 * ks + khi) * 16), f.k[ks]);
#pragma unroll
    for (int mt = 0; mt < MmaFrags<Cfg>::MT; ++mt)
      ldsm_x4_trans(vb + tile_off<ROWB>(vtok, (2 * mt + vhi) * 16), f.v[mt]);
  }
}

template <class Cfg>
__device__ __forceinline__ void mma_compute(MmaState<Cfg> &st, const MmaFrags<Cfg> &f, const DecodeParams &p,
                                            const StageMeta &m, int lane) {
  static_assert(MmaState<Cfg>::NH == 1, "one-block steps serve 8-row units");
  constexpr bool kBF = (Cfg::Cache::kCode == PKV_BF16);
  const int gid = lane >> 2;
  // token rows r of the block visible to score column c: base_c <= r < base_c + W,
  // base_c = rem - back_c - W (one unsigned compare; W = 2^30 without a window)
  const int base0 = m.rem - st.back[0][0] - p.wlen, base1 = m.rem - st.back[0][1] - p.wlen;
  const uint32_t wl = (uint32_t)p.wlen;

  // ---- scores S^T = K . Q^T (16 tokens x 8 rows), two independent chains ----
  float s[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int ks = 0; ks < MmaFrags<Cfg>::KS; ++ks) {
    uint32_t a[4];
    if constexpr (Cfg::FP8) {
      // k-slots 2t,2t+1 | 2t+8,2t+9 of row gid (+8) hold d = 16ks + 4t + {0,1} | {2,3}
      a[0] = e4m3x2_to_f16x2((uint16_t)(f.k[ks][0] & 0xffff));
      a[1] = e4m3x2_to_f16x2((uint16_t)(f.k[ks][1] & 0xffff));
      a[2] = e4m3x2_to_f16x2((uint16_t)(f.k[ks][0] >> 16));
      a[3] = e4m3x2_to_f16x2((uint16_t)(f.k[ks][1] >> 16));
    } else {
      a[0] = f.k[ks][0]; a[1] = f.k[ks][1]; a[2] = f.k[ks][2]; a[3] = f.k[ks][3];
    }
    if (ks & 1)
      mma16816<kBF>(s1, a, st.qb[0][ks][0], st.qb[0][ks][1]);
    else
      mma16816<kBF>(s, a, st.qb[0][ks][0], st.qb[0][ks][1]);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) s[i] += s1[i];

  // ---- online softmax over the block (log2 domain) ----
  const float sc = p.scale_log2 * m.ks;
  float x0 = s[0] * sc, x1 = s[1] * sc, x2 = s[2] * sc, x3 = s[3] * sc;
  if ((uint32_t)(gid - base0) >= wl) x0 = -INFINITY;
  if ((uint32_t)(gid - base1) >= wl) x1 = -INFINITY;
  if ((uint32_t)(gid + 8 - base0) >= wl) x2 = -INFINITY;
  if ((uint32_t)(gid + 8 - base1) >= wl) x3 = -INFINITY;
  float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
  // the running maxima change only when some lane holds a larger score;
  // otherwise the exchange and the rescale (by exactly 1) are skipped
  if (__any_sync(kFull, (mx0 > st.m[0][0]) | (mx1 > st.m[0][1]))) {
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, off));
    }
    const float mn0 = fmaxf(st.m[0][0], mx0), mn1 = fmaxf(st.m[0][1], mx1);
    // a column that has seen no visible position yet keeps weight 0 (not NaN)
    const float nb0 = mn0 == -INFINITY ? 0.f : mn0, nb1 = mn1 == -INFINITY ? 0.f : mn1;
    const float al0 = exp2f(st.m[0][0] - nb0), al1 = exp2f(st.m[0][1] - nb1);
    st.l[0][0] *= al0;
    st.l[0][1] *= al1;
    st.m[0][0] = mn0;
    st.m[0][1] = mn1;
#pragma unroll
    for (int mt = 0; mt < MmaFrags<Cfg>::MT; ++mt) {
      st.acc[0][mt][0] *= al0;
      st.acc[0][mt][1] *= al1;
      st.acc[0][mt][2] *= al0;
      st.acc[0][mt][3] *= al1;
    }
  }
  const float mb0 = st.m[0][0] == -INFINITY ? 0.f : st.m[0][0];
  const float mb1 = st.m[0][1] == -INFINITY ? 0.f : st.m[0][1];
  const float p0 = exp2f(x0 - mb0), p1 = exp2f(x1 - mb1);
  const float p2 = exp2f(x2 - mb0), p3 = exp2f(x3 - mb1);
  st.l[0][0] += p0 + p2;
  st.l[0][1] += p1 + p3;

  // ---- O^T += V^T . P^T ----
  if constexpr (Cfg::FP8) {
    const float vs = m.vs;  // fold the V scale into the weights
    const uint32_t pb0 = movmatrix_trans(pack_f16x2(p0 * vs, p1 * vs));
    const uint32_t pb1 = movmatrix_trans(pack_f16x2(p2 * vs, p3 * vs));
#pragma unroll
    for (int mt = 0; mt < MmaFrags<Cfg>::MT; ++mt) {
      // bytes 2mt, 2mt+1 of the thread's head-dim run, from token rows
      // (2t, 2t+1) and (2t+8, 2t+9), paired for the f16x2 conversion
      const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;
      const uint32_t x = __byte_perm(f.v[0][mt >> 1], f.v[1][mt >> 1], sel);
      const uint32_t y = __byte_perm(f.v[2][mt >> 1], f.v[3][mt >> 1], sel);
      uint32_t a[4];
      a[0] = e4m3x2_to_f16x2((uint16_t)(x & 0xffff));
      a[1] = e4m3x2_to_f16x2((uint16_t)(x >> 16));
      a[2] = e4m3x2_to_f16x2((uint16_t)(y & 0xffff));
      a[3] = e4m3x2_to_f16x2((uint16_t)(y >> 16));
      mma16816<false>(st.acc[0][mt], a, pb0, pb1);
    }
  } else if constexpr (kBF) {
    // bf16 keeps 8 significant bits; short contexts give weights near 1
    // whose rounding would show in the output, so P goes in as a bf16 high
    // part plus a bf16 residual (two MMAs on the same V fragments)
    const __nv_bfloat162 h01 = __floats2bfloat162_rn(p0, p1), h23 = __floats2bfloat162_rn(p2, p3);
    const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
    const uint32_t pb0 = movmatrix_trans(*reinterpret_cast<const uint32_t *>(&h01));
    const uint32_t pb1 = movmatrix_trans(*reinterpret_cast<const uint32_t *>(&h23));
    const uint32_t lb0 = movmatrix_trans(pack_bf16x2(p0 - f01.x, p1 - f01.y));
    const uint32_t lb1 = movmatrix_trans(pack_bf16x2(p2 - f23.x, p3 - f23.y));
#pragma unroll
    for (int mt = 0; mt < MmaFrags<Cfg>::MT; ++mt) {
      mma16816<true>(st.acc[0][mt], f.v[mt], pb0, pb1);
      mma16816<true>(st.acc[0][mt], f.v[mt], lb0, lb1);
    }
  } else {
    const uint32_t pb0 = movmatrix_trans(pack_f16x2(p0, p1));
    const uint32_t pb1 = movmatrix_trans(pack_f16x2(p2, p3));
#pragma unroll
    for (int mt = 0; mt < MmaFrags<Cfg>::MT; ++mt) mma16816<false>(st.acc[0][mt], f.v[mt], pb0, pb1);
  }
}

// ---------------------------------------------------------------------------
// Two-block stages (fp8 caches): the same arithmetic as mma_load /
// mma_compute, over the 32 tokens of two consecutive blocks of one unit with
// one online-softmax update.  K fragments are loaded and consumed before the
// V fragments, which keeps the register footprint of two blocks in bounds.
// ---------------------------------------------------------------------------
// S^T = K . Q^T of one fp8 block for every 8-row group of the unit (two
// independent MMA chains per group, summed); each K fragment is widened once
// for all groups.
template <class Cfg>
__device__ __forceinline__ void fp8_scores(const MmaState<Cfg> &st, const uint8_t *tk, int lane,
                                           float (&s)[MmaState<Cfg>::NH][4]) {
  constexpr int ROWB = Cfg::ROWB, NH = MmaState<Cfg>::NH;
  const int gid = lane >> 2, tig = lane & 3;
  const uint32_t kb = smem_u32(tk);
  float s0[NH][4], s1[NH][4];
#pragma unroll
  for (int nh = 0; nh < NH; ++nh)
#pragma unroll
    for (int i = 0; i < 4; ++i) s0[nh][i] = s1[nh][i] = 0.f;
#pragma unroll
  for (int ks = 0; ks < MmaState<Cfg>::KS; ++ks) {
    // k-slots 2t,2t+1 | 2t+8,2t+9 of row gid (+8) hold d = 16ks + 4t + {0,1} | {2,3}
    const uint32_t k0 = lds32(kb + tile_off<ROWB>(gid, 16 * ks + 4 * tig));
    const uint32_t k1 = lds32(kb + tile_off<ROWB>(gid + 8, 16 * ks + 4 * tig));
    uint32_t a[4];
    a[0] = e4m3x2_to_f16x2((uint16_t)(k0 & 0xffff));
    a[1] = e4m3x2_to_f16x2((uint16_t)(k1 & 0xffff));
    a[2] = e4m3x2_to_f16x2((uint16_t)(k0 >> 16));
    a[3] = e4m3x2_to_f16x2((uint16_t)(k1 >> 16));
#pragma unroll
    for (int nh = 0; nh < NH; ++nh) {
      // one chain per column group when there are two groups (the groups'
      // chains interleave); an 8-row unit alternates two chains
      if (NH == 1 && (ks & 1))
        mma16816<false>(s1[nh], a, st.qb[nh][ks][0], st.qb[nh][ks][1]);
      else
        mma16816<false>(s0[nh], a, st.qb[nh][ks][0], st.qb[nh][ks][1]);
    }
  }
#pragma unroll
  for (int nh = 0; nh < NH; ++nh)
#pragma unroll
    for (int i = 0; i < 4; ++i) s[nh][i] = NH == 1 ? s0[nh][i] + s1[nh][i] : s0[nh][i];
}

// O^T += V^T . P^T of one fp8 block for every 8-row group, P (with the
// block's V scale folded in) already in B-operand form; each V fragment is
// widened once for all groups.
template <class Cfg>
__device__ __forceinline__ void fp8_pv(MmaState<Cfg> &st, const uint8_t *tv, int lane,
                                       const uint32_t (&pb)[MmaState<Cfg>::NH][2]) {
  constexpr int ROWB = Cfg::ROWB, NH = MmaState<Cfg>::NH;
  constexpr int DPT = Cfg::D / 8;  // head-dim bytes owned by one row group
  const int gid = lane >> 2, tig = lane & 3;
  const uint32_t vb = smem_u32(tv);
  const int trow[4] = {2 * tig, 2 * tig + 1, 2 * tig + 8, 2 * tig + 9};
  uint32_t v[4][DPT / 4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (DPT == 16) {
      const uint4 r = lds128(vb + tile_off<ROWB>(trow[i], 16 * gid));
      v[i][0] = r.x; v[i][1] = r.y; v[i][2] = r.z; v[i][3] = r.w;
    } else {
      const uint2 r = lds64(vb + tile_off<ROWB>(trow[i], 8 * gid));
      v[i][0] = r.x; v[i][1] = r.y;
    }
  }
#pragma unroll
  for (int mt = 0; mt < MmaState<Cfg>::MT; ++mt) {
    // bytes 2mt, 2mt+1 of the thread's head-dim run, from token rows
    // (2t, 2t+1) and (2t+8, 2t+9), paired for the f16x2 conversion
    const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;
    const uint32_t x = __byte_perm(v[0][mt >> 1], v[1][mt >> 1], sel);
    const uint32_t y = __byte_perm(v[2][mt >> 1], v[3][mt >> 1], sel);
    uint32_t a[4];
    a[0] = e4m3x2_to_f16x2((uint16_t)(x & 0xffff));
    a[1] = e4m3x2_to_f16x2((uint16_t)(x >> 16));
    a[2] = e4m3x2_to_f16x2((uint16_t)(y & 0xffff));
    a[3] = e4m3x2_to_f16x2((uint16_t)(y >> 16));
#pragma unroll
    for (int nh = 0; nh < NH; ++nh) mma16816<false>(st.acc[nh][mt], a, pb[nh][0], pb[nh][1]);
  }
}

template <class Cfg>
__device__ __forceinline__ void mma_pair(MmaState<Cfg> &st, const DecodeParams &p, const StageMeta &m,
                                         uint8_t *tk0, int lane) {
  static_assert(Cfg::FP8, "two-block stages are the fp8 path");
  constexpr int ROWB = Cfg::ROWB, NH = MmaState<Cfg>::NH;
  const int gid = lane >> 2;
  const bool two = m.nb == 2;
  uint8_t *tv0 = tk0 + Cfg::TILE, *tk1 = tk0 + 2 * Cfg::TILE, *tv1 = tk0 + 3 * Cfg::TILE;
  const int rem0 = m.rem, rem1 = m.rem - kBlock;
  if (rem0 < kBlock) zero_tail_rows<ROWB>(tv0, rem0, lane);
  if (two && rem1 < kBlock) zero_tail_rows<ROWB>(tv1, rem1, lane);

  float s[NH][4], t[NH][4];
  fp8_scores<Cfg>(st, tk0, lane, s);
  if (two) fp8_scores<Cfg>(st, tk1, lane, t);

  const uint32_t wl = (uint32_t)p.wlen;
  const float sc0 = p.scale_log2 * m.ks, sc1 = p.scale_log2 * m.ks1;
  // 16-row units: when every row of the stage is visible to every column of
  // the unit (the common case: not the last blocks of a context, no window
  // edge inside) no mask is applied — warp-uniform, from the stage's position
  // and the unit's row limits.  (Measured: +4 % for 16-row units; the 8-row
  // units, with half the mask work per stage, keep the masks.)
  const bool full = NH > 1 && rem0 - st.bk_hi >= (two ? 2 * kBlock : kBlock) && rem0 - st.bk_lo <= p.wlen;
  uint32_t pa[NH][2], pc[NH][2];  // B operands of the first and second block
#pragma unroll
  for (int nh = 0; nh < NH; ++nh) {
    float x0 = s[nh][0] * sc0, x1 = s[nh][1] * sc0, x2 = s[nh][2] * sc0, x3 = s[nh][3] * sc0;
    float y0 = -INFINITY, y1 = -INFINITY, y2 = -INFINITY, y3 = -INFINITY;
    if (two) {
      y0 = t[nh][0] * sc1; y1 = t[nh][1] * sc1; y2 = t[nh][2] * sc1; y3 = t[nh][3] * sc1;
    }
    if (!full) {
      // token rows r of a block visible to score column c: base_c <= r < base_c + W
      // (see mma_compute); the second block's base is 16 lower
      const int base0 = rem0 - st.back[nh][0] - p.wlen, base1 = rem0 - st.back[nh][1] - p.wlen;
      if ((uint32_t)(gid - base0) >= wl) x0 = -INFINITY;
      if ((uint32_t)(gid - base1) >= wl) x1 = -INFINITY;
      if ((uint32_t)(gid + 8 - base0) >= wl) x2 = -INFINITY;
      if ((uint32_t)(gid + 8 - base1) >= wl) x3 = -INFINITY;
      if ((uint32_t)(gid + 16 - base0) >= wl) y0 = -INFINITY;
      if ((uint32_t)(gid + 16 - base1) >= wl) y1 = -INFINITY;
      if ((uint32_t)(gid + 24 - base0) >= wl) y2 = -INFINITY;
      if ((uint32_t)(gid + 24 - base1) >= wl) y3 = -INFINITY;
    }
    float mx0 = fmaxf(fmaxf(x0, x2), fmaxf(y0, y2)), mx1 = fmaxf(fmaxf(x1, x3), fmaxf(y1, y3));
    // The running maxima change only when some lane holds a larger score;
    // otherwise (16-row units) the column maxima, the rescale (a factor of
    // exactly 1) and the max exchange are skipped (warp-uniform vote).  The
    // 8-row units always exchange: the vote measured slower there.
    if (NH == 1 || __any_sync(kFull, (mx0 > st.m[nh][0]) | (mx1 > st.m[nh][1]))) {
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, off));
      }
      const float mn0 = fmaxf(st.m[nh][0], mx0), mn1 = fmaxf(st.m[nh][1], mx1);
      // a column that has seen no visible position yet keeps weight 0 (not NaN)
      const float nb0 = mn0 == -INFINITY ? 0.f : mn0, nb1 = mn1 == -INFINITY ? 0.f : mn1;
      const float al0 = exp2f(st.m[nh][0] - nb0), al1 = exp2f(st.m[nh][1] - nb1);
      st.l[nh][0] *= al0;
      st.l[nh][1] *= al1;
      st.m[nh][0] = mn0;
      st.m[nh][1] = mn1;
#pragma unroll
      for (int mt = 0; mt < MmaState<Cfg>::MT; ++mt) {
        st.acc[nh][mt][0] *= al0;
        st.acc[nh][mt][1] *= al1;
        st.acc[nh][mt][2] *= al0;
        st.acc[nh][mt][3] *= al1;
      }
    }
    const float mb0 = st.m[nh][0] == -INFINITY ? 0.f : st.m[nh][0];
    const float mb1 = st.m[nh][1] == -INFINITY ? 0.f : st.m[nh][1];
    const float p0 = exp2f(x0 - mb0), p1 = exp2f(x1 - mb1), p2 = exp2f(x2 - mb0), p3 = exp2f(x3 - mb1);
    const float q0 = exp2f(y0 - mb0), q1 = exp2f(y1 - mb1), q2 = exp2f(y2 - mb0), q3 = exp2f(y3 - mb1);
    st.l[nh][0] += (p0 + p2) + (q0 + q2);
    st.l[nh][1] += (p1 + p3) + (q1 + q3);
    // the V scales folded into the weights
    pa[nh][0] = movmatrix_trans(pack_f16x2(p0 * m.vs, p1 * m.vs));
    pa[nh][1] = movmatrix_trans(pack_f16x2(p2 * m.vs, p3 * m.vs));
    pc[nh][0] = movmatrix_trans(pack_f16x2(q0 * m.vs1, q1 * m.vs1));
    pc[nh][1] = movmatrix_trans(pack_f16x2(q2 * m.vs1, q3 * m.vs1));
  }
  fp8_pv<Cfg>(st, tv0, lane, pa);
  if (two) fp8_pv<Cfg>(st, tv1, lane, pc);
}

// Head-dim index held by accumulator row group `r` (0: gid, 1: gid + 8) of m-tile mt.
template <class Cfg>
__device__ __forceinline__ int mma_dim(int mt, int r, int gid) {
  if constexpr (Cfg::FP8)
    return gid * (Cfg::D / 8) + 2 * mt + r;
  else
    return 16 * mt + gid + 8 * r;
}

template <class Cfg>
__device__ __forceinline__ void mma_finish(MmaState<Cfg> &st, const DecodeParams &p, const StageMeta &m,
                                           int w, int lane) {
  const int gid = lane >> 2, tig = lane & 3;
  const int h = m.hu / p.NC, r0 = (m.hu % p.NC) * Cfg::GC;
  const int gc = min(Cfg::GC, p.R - r0);
  const bool complete = m.flags & kComplete;
  // partials: [worker][slot][GC rows][D]
  const size_t base = ((size_t)w * 2 + ((m.flags & kWFirst) ? 0 : 1)) * Cfg::GC;
#pragma unroll
  for (int nh = 0; nh < MmaState<Cfg>::NH; ++nh) {
    float l0 = st.l[nh][0], l1 = st.l[nh][1];
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0 += __shfl_xor_sync(kFull, l0, off);
      l1 += __shfl_xor_sync(kFull, l1, off);
    }
    // a row with no visible position (context shorter than q_len) gives 0
    const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
    const int hA = 8 * nh + 2 * tig, hB = hA + 1;
    if (complete) {
      const size_t baseA = hA < gc ? query_row(p, m.b, h, r0 + hA) : 0;
      const size_t baseB = hB < gc ? query_row(p, m.b, h, r0 + hB) : 0;
#pragma unroll
      for (int mt = 0; mt < MmaState<Cfg>::MT; ++mt)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int d = mma_dim<Cfg>(mt, r, gid);
          if (hA < gc) store_scalar(typename Cfg::Q{}, p.out, baseA + d, st.acc[nh][mt][2 * r] * inv0);
          if (hB < gc) store_scalar(typename Cfg::Q{}, p.out, baseB + d, st.acc[nh][mt][2 * r + 1] * inv1);
        }
    } else {
      float *oA = p.part_o + (base + hA) * Cfg::D;
      float *oB = p.part_o + (base + hB) * Cfg::D;
#pragma unroll
      for (int mt = 0; mt < MmaState<Cfg>::MT; ++mt)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int d = mma_dim<Cfg>(mt, r, gid);
          if (hA < gc) oA[d] = st.acc[nh][mt][2 * r] * inv0;
          if (hB < gc) oB[d] = st.acc[nh][mt][2 * r + 1] * inv1;
        }
      if (gid == 0) {
        if (hA < gc) p.part_lse[base + hA] = st.m[nh][0] + log2f(l0);
        if (hB < gc) p.part_lse[base + hB] = st.m[nh][1] + log2f(l1);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// CUDA-core path state and steps (GC in {1, 2}).
// ---------------------------------------------------------------------------
template <class Cfg>
struct SimtState {
  static constexpr int DPL = Cfg::D / 32;  // head-dim elements per lane in p.V
  float acc[Cfg::GC][DPL];
  float m[Cfg::GC], l[Cfg::GC];
  int back[Cfg::GC];
};

// 16 bytes of cache elements -> floats
template <class T>
__device__ __forceinline__ void cvt16(T, const uint4 &raw, float *f);
template <>
__device__ __forceinline__ void cvt16(F32, const uint4 &raw, float *f) {
  f[0] = __uint_as_float(raw.x); f[1] = __uint_as_float(raw.y);
  f[2] = __uint_as_float(raw.z); f[3] = __uint_as_float(raw.w);
}
template <>
__device__ __forceinline__ void cvt16(F16, const uint4 &raw, float *f) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) { const float2 v = unpack2(F16{}, w[i]); f[2 * i] = v.x; f[2 * i + 1] = v.y; }
}
template <>
__device__ __forceinline__ void cvt16(BF16, const uint4 &raw, float *f) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) { const float2 v = unpack2(BF16{}, w[i]); f[2 * i] = v.x; f[2 * i + 1] = v.y; }
}
template <>
__device__ __forceinline__ void cvt16(E4M3, const uint4 &raw, float *f) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 a = unpack2_e4m3((uint16_t)(w[i] & 0xffff));
    const float2 b = unpack2_e4m3((uint16_t)(w[i] >> 16));
    f[4 * i] = a.x; f[4 * i + 1] = a.y; f[4 * i + 2] = b.x; f[4 * i + 3] = b.y;
  }
}

// DPL elements of one V row owned by a lane -> floats
template <class Cfg>
__device__ __forceinline__ void load_vrow(uint32_t addr, float *f) {
  using T = typename Cfg::Cache;
  constexpr int DPL = SimtState<Cfg>::DPL;
  constexpr int BYTES = DPL * T::kBytes;
  if constexpr (BYTES == 16) {
    cvt16(T{}, lds128(addr), f);
  } else if constexpr (BYTES == 8) {
    const uint2 v = lds64(addr);
    if constexpr (T::kCode == PKV_F32) {
      f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
    } else {
      const float2 a = unpack2(T{}, v.x), b = unpack2(T{}, v.y);
      f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    }
  } else if constexpr (BYTES == 4) {
    const uint32_t v = lds32(addr);
    if constexpr (T::kCode == PKV_FP8_E4M3) {
      const float2 a = unpack2_e4m3((uint16_t)(v & 0xffff)), b = unpack2_e4m3((uint16_t)(v >> 16));
      f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    } else {
      const float2 a = unpack2(T{}, v);
      f[0] = a.x; f[1] = a.y;
    }
  } else {  // 2 bytes: two e4m3 values
    const float2 a = unpack2_e4m3((uint16_t)lds16(addr));
    f[0] = a.x; f[1] = a.y;
  }
}

template <class Cfg>
__device__ __forceinline__ void simt_begin(SimtState<Cfg> &st, const DecodeParams &p, const StageMeta &m,
                                           float *qbuf, int lane) {
  const int h = m.hu / p.NC, r0 = (m.hu % p.NC) * Cfg::GC;
  const int gc = min(Cfg::GC, p.R - r0);
  __syncwarp();
  for (int idx = lane; idx < Cfg::GC * Cfg::D; idx += 32) {
    const int g = idx / Cfg::D, d = idx % Cfg::D;
    qbuf[idx] = g < gc ? load_scalar(typename Cfg::Q{}, p.q, query_row(p, m.b, h, r0 + g) + d) : 0.f;
  }
  __syncwarp();
#pragma unroll
  for (int g = 0; g < Cfg::GC; ++g) {
    st.back[g] = row_back(p, r0 + g);
    st.m[g] = -INFINITY;
    st.l[g] = 0.f;
#pragma unroll
    for (int e = 0; e < SimtState<Cfg>::DPL; ++e) st.acc[g][e] = 0.f;
  }
}

template <class Cfg>
__device__ __forceinline__ void simt_block(SimtState<Cfg> &st, const DecodeParams &p, const StageMeta &m,
                                           uint8_t *tk, uint8_t *tv, const float *qbuf, int lane) {
  using T = typename Cfg::Cache;
  constexpr int GC = Cfg::GC, D = Cfg::D, ROWB = Cfg::ROWB;
  constexpr int HB = ROWB / 2;            // bytes of half a row
  constexpr int EPC = 16 / T::kBytes;     // elements per 16-byte chunk
  constexpr int DPL = SimtState<Cfg>::DPL;
  const uint32_t kb = smem_u32(tk), vb = smem_u32(tv);
  const int t = lane & 15, half = lane >> 4;
  const int nvalid = m.nvalid;
  int vis = 0;  // rows visible to some column: p.V skips the rest
#pragma unroll
  for (int g = 0; g < GC; ++g) vis = max(vis, min(nvalid, m.rem - st.back[g]));

  // scores: lane (t, half) dots token t with half of q, then the halves add
  float part[GC];
#pragma unroll
  for (int g = 0; g < GC; ++g) part[g] = 0.f;
#pragma unroll
  for (int i = 0; i < HB / 16; ++i) {
    float kf[EPC];
    cvt16(T{}, lds128(kb + tile_off<ROWB>(t, half * HB + 16 * i)), kf);
    const float *qp = qbuf + half * (D / 2) + i * EPC;
#pragma unroll
    for (int g = 0; g < GC; ++g)
#pragma unroll
      for (int e = 0; e < EPC; e += 4) {
        const float4 qv = *reinterpret_cast<const float4 *>(qp + g * D + e);
        part[g] = fmaf(qv.x, kf[e], part[g]);
        part[g] = fmaf(qv.y, kf[e + 1], part[g]);
        part[g] = fmaf(qv.z, kf[e + 2], part[g]);
        part[g] = fmaf(qv.w, kf[e + 3], part[g]);
      }
  }
  const float sc = p.scale_log2 * m.ks;
  float pw[GC];
#pragma unroll
  for (int g = 0; g < GC; ++g) {
    float x = part[g] + __shfl_xor_sync(kFull, part[g], 16);
    x = ((uint32_t)(t - (m.rem - st.back[g] - p.wlen)) < (uint32_t)p.wlen) ? x * sc : -INFINITY;
    float bm = x;
#pragma unroll
    for (int off = 1; off < 16; off <<= 1) bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, off));
    const float mn = fmaxf(st.m[g], bm);
    const float mb = mn == -INFINITY ? 0.f : mn;  // no visible position yet: weight 0
    const float al = exp2f(st.m[g] - mb);
    const float pg = exp2f(x - mb);
    float bs = pg;
#pragma unroll
    for (int off = 1; off < 16; off <<= 1) bs += __shfl_xor_sync(kFull, bs, off);
    st.l[g] = st.l[g] * al + bs;
    st.m[g] = mn;
    pw[g] = pg * m.vs;
#pragma unroll
    for (int e = 0; e < DPL; ++e) st.acc[g][e] *= al;
  }
  // p.V: lane owns head-dim elements [lane*DPL, lane*DPL + DPL)
  const uint32_t vcol = lane * DPL * T::kBytes;
  for (int tt = 0; tt < vis; ++tt) {
    float vf[DPL];
    load_vrow<Cfg>(vb + tile_off<ROWB>(tt, vcol), vf);
#pragma unroll
    for (int g = 0; g < GC; ++g) {
      const float pt = __shfl_sync(kFull, pw[g], tt);
#pragma unroll
      for (int e = 0; e < DPL; ++e) st.acc[g][e] = fmaf(pt, vf[e], st.acc[g][e]);
    }
  }
}

template <class Cfg>
__device__ __forceinline__ void simt_finish(SimtState<Cfg> &st, const DecodeParams &p, const StageMeta &m,
                                            int w, int lane) {
  constexpr int DPL = SimtState<Cfg>::DPL;
  const int h = m.hu / p.NC, r0 = (m.hu % p.NC) * Cfg::GC;
  const int gc = min(Cfg::GC, p.R - r0);
  if (m.flags & kComplete) {
#pragma unroll
    for (int g = 0; g < Cfg::GC; ++g) {
      if (g >= gc) break;
      const float inv = st.l[g] > 0.f ? 1.f / st.l[g] : 0.f;
      const size_t base = query_row(p, m.b, h, r0 + g) + lane * DPL;
#pragma unroll
      for (int e = 0; e < DPL; ++e) store_scalar(typename Cfg::Q{}, p.out, base + e, st.acc[g][e] * inv);
    }
  } else {
    const int slot = (m.flags & kWFirst) ? 0 : 1;
    const size_t base = ((size_t)w * 2 + slot) * Cfg::GC;  // [worker][slot][GC rows][D]
#pragma unroll
    for (int g = 0; g < Cfg::GC; ++g) {
      if (g >= gc) break;
      const float inv = st.l[g] > 0.f ? 1.f / st.l[g] : 0.f;
      float *o = p.part_o + (base + g) * Cfg::D + lane * DPL;
#pragma unroll
      for (int e = 0; e < DPL; ++e) o[e] = st.acc[g][e] * inv;
      if (lane == 0) p.part_lse[base + g] = st.m[g] + log2f(st.l[g]);
    }
  }
}

// ---------------------------------------------------------------------------
// Inline plan (batches of up to kInlinePrefix - 1 sequences): every CTA scans
// context_lens into a shared-memory prefix of blocks per sequence,
// prefix[b] = sum_{b' < b} items_b' (seq_items: blocks inside the windows), so no separate plan launch is
// needed; CTA 0 also stores it for the merge kernel.  Lengths are clamped to
// [0, 16 * max_blocks] and flagged.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int clamp_len(const DecodeParams &p, int ctx, int *flags) {
  if (ctx < 0 || ctx > p.max_blocks * kBlock) *flags |= PKV_FLAG_BAD_LEN;
  return clamped_len(p, ctx);
}

__device__ __forceinline__ void inline_plan(const DecodeParams &p, int32_t *s_prefix, int32_t *s_scan,
                                            int *cta_flags) {
  const int T = blockDim.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nw = T >> 5;
  const int k = (p.B + T - 1) / T;  // consecutive sequences per thread
  const int b0 = tid * k;
  int sum = 0, flags = 0;
  for (int i = 0; i < k; ++i)
    if (b0 + i < p.B) sum += seq_items(p, clamp_len(p, __ldg(p.context_lens + b0 + i), &flags));
  int x = sum;  // inclusive scan within the warp
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(kFull, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) s_scan[wid] = x;
  __syncthreads();
  if (wid == 0) {
    const int v = lane < nw ? s_scan[lane] : 0;
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(kFull, incl, off);
      if (lane >= off) incl += y;
    }
    if (lane < nw) s_scan[lane] = incl - v;
  }
  __syncthreads();
  int run = s_scan[wid] + x - sum;
  int unused = 0;
  for (int i = 0; i < k; ++i) {
    const int b = b0 + i;
    if (b < p.B) {
      s_prefix[b] = run;
      run += seq_items(p, clamp_len(p, __ldg(p.context_lens + b), &unused));
      if (b == p.B - 1) s_prefix[p.B] = run;
    }
  }
  if (flags) atomicOr(cta_flags, flags);
  __syncthreads();
  if (blockIdx.x == 0)
    for (int b = tid; b <= p.B; b += T) p.prefix[b] = s_prefix[b];
}

// Partition w's first item {s, b, hu, j} and its end, from the prefix.
__device__ __forceinline__ int4 locate(const DecodeParams &p, const int32_t *pre, int w, int *end) {
  const int64_t W = (int64_t)p.HU * pre[p.B];
  const int64_t Pe = active_partitions(p, W);
  const int64_t s = w < Pe ? W * w / Pe : W;
  *end = w < Pe ? (int)(W * (w + 1) / Pe) : (int)W;
  if (s >= W) return make_int4((int)W, p.B, 0, 0);
  int lo = 0, hi = p.B - 1;  // largest b with HU * prefix[b] <= s
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((int64_t)p.HU * pre[mid] <= s)
      lo = mid;
    else
      hi = mid - 1;
  }
  const int n = pre[lo + 1] - pre[lo];
  const int64_t rr = s - (int64_t)p.HU * pre[lo];
  const int j0 = first_block(p, clamped_len(p, __ldg(p.context_lens + lo)));
  return make_int4((int)s, lo, (int)(rr / n), j0 + (int)(rr % n));
}

// ---------------------------------------------------------------------------
// The kernel.
// ---------------------------------------------------------------------------
template <class Cfg>
__global__ void __launch_bounds__(Cfg::WARPS * 32, Cfg::MIN_CTAS)
    decode_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the 128-byte swizzle, by pointer arithmetic on the
  // shared array so every access stays a shared-memory access
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  uint8_t *tiles = smem + (size_t)wib * Cfg::STAGES * Cfg::STAGE_BYTES;
  StageMeta *meta = reinterpret_cast<StageMeta *>(smem + Cfg::TILES_BYTES) + wib * Cfg::STAGES;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::TILES_BYTES + Cfg::META_BYTES) + wib * Cfg::STAGES;
  float *qbuf = reinterpret_cast<float *>(smem + Cfg::TILES_BYTES + Cfg::META_BYTES + Cfg::BAR_BYTES) +
                wib * Cfg::GC * Cfg::D;
  int32_t *s_prefix =
      reinterpret_cast<int32_t *>(smem + Cfg::TILES_BYTES + Cfg::META_BYTES + Cfg::BAR_BYTES + Cfg::QBUF_BYTES);
  __shared__ int32_t s_scan[32];
  __shared__ int cta_flags;
  __shared__ __align__(8) uint64_t dead_bar;  // failure-path test hook: nothing ever arrives on it
  if (threadIdx.x == 0) cta_flags = 0;
  if (lane == 0) {
    for (int s = 0; s < Cfg::STAGES; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
  }
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  __syncwarp();
  grid_dep_wait();  // the previous kernel's writes are visible from here on
  if (p.inline_plan) inline_plan(p, s_prefix, s_scan, &cta_flags);

  const int w = blockIdx.x * Cfg::WARPS + wib;
  if (w < p.P) {
    int e;
    int4 st0;
    if (p.inline_plan) {
      st0 = locate(p, s_prefix, w, &e);
    } else {
      st0 = p.starts[w];
      e = p.starts[w + 1].x;
    }
    const int total = e - st0.x;
    // Failure-path test hook: the worker holding the first work item replaces
    // its first pipeline wait by a wait on dead_bar, which runs out and takes
    // the timeout path below.
    const bool stall = p.stall_ns != 0 && st0.x == 0 && total > 0;
    if (stall) {
      if (lane == 0) {
        mbar_init(&dead_bar, 1);
        fence_barrier_init();
      }
      __syncwarp();
    }
    if (total > 0) {
      Producer pr;
      pr.pi = st0.x;
      pr.e = e;
      pr.s = st0.x;
      pr.b = st0.y;
      pr.hu = st0.z;
      pr.j = st0.w;
      pr.seg_j0 = 0;
      pr.seg_wfirst = 0;
      pr.win_b = -1;
      pr.win_hu = -1;
      pr.win_j0 = 0;
      pr.win_id = 0;
      pr.win_ks = pr.win_vs = 0.f;
      load_seq(pr, p);
      if constexpr (Cfg::BPS == 2) {
        // two-block stages: items issued / consumed are counted apart from
        // the stages that carry them
        int issued = 0, nst = 0;
        for (; nst < Cfg::STAGES && issued < total; ++nst)
          issued += produce<Cfg>(pr, p, &tmK, &tmV, tiles, meta, bars, nst, lane, &cta_flags);
        MmaState<Cfg> state;
        for (int done = 0, i = 0; done < total; ++i) {
          const int stage = i % Cfg::STAGES;
          const uint32_t parity = (uint32_t)(i / Cfg::STAGES) & 1u;
          if ((stall && i == 0) ? !mbar_wait_bounded(&dead_bar, 0, p.timeout_ns)
                                : !mbar_wait_bounded(&bars[stage], parity, p.timeout_ns)) {
            if (lane == 0) atomicOr(&cta_flags, PKV_FLAG_TIMEOUT);
            // let the copies still in flight land before the CTA's memory goes away
            for (int k = i; k < nst; ++k)
              mbar_wait_bounded(&bars[k % Cfg::STAGES], (uint32_t)(k / Cfg::STAGES) & 1u, p.timeout_ns);
            break;
          }
          const StageMeta m = meta[stage];
          if (m.flags & kFirst) mma_begin<Cfg>(state, p, m, lane);
          mma_pair<Cfg>(state, p, m, tiles + (size_t)stage * Cfg::STAGE_BYTES, lane);
          if (issued < total) {  // refilled once its fragments are consumed (as below)
            issued += produce<Cfg>(pr, p, &tmK, &tmV, tiles, meta, bars, stage, lane, &cta_flags);
            ++nst;
          }
          if (m.flags & kLast) mma_finish<Cfg>(state, p, m, w, lane);
          done += m.nb;
        }
      } else {
      int issued = 0;
      for (; issued < Cfg::STAGES && issued < total; ++issued)
        produce<Cfg>(pr, p, &tmK, &tmV, tiles, meta, bars, issued, lane, &cta_flags);

      typename std::conditional<Cfg::MMA, MmaState<Cfg>, SimtState<Cfg>>::type state;
      for (int i = 0; i < total; ++i) {
        const int stage = i % Cfg::STAGES;
        const uint32_t parity = (uint32_t)(i / Cfg::STAGES) & 1u;
        if ((stall && i == 0) ? !mbar_wait_bounded(&dead_bar, 0, p.timeout_ns)
                              : !mbar_wait_bounded(&bars[stage], parity, p.timeout_ns)) {
          if (lane == 0) atomicOr(&cta_flags, PKV_FLAG_TIMEOUT);
          // let the copies still in flight land before the CTA's memory goes away
          for (int k = i; k < issued; ++k)
            mbar_wait_bounded(&bars[k % Cfg::STAGES], (uint32_t)(k / Cfg::STAGES) & 1u, p.timeout_ns);
          break;
        }
        const StageMeta m = meta[stage];
        uint8_t *tk = tiles + (size_t)stage * Cfg::STAGE_BYTES;
        uint8_t *tv = tk + Cfg::TILE;
        if constexpr (Cfg::MMA) {
          // The stage is refilled after the block is computed: every fragment
          // has been consumed by then, so the TMA overwrite needs no proxy
          // fence.  (Refilling it right after the fragments reach registers
          // measured 1-2 % slower on GB300.)
          if (m.flags & kFirst) mma_begin<Cfg>(state, p, m, lane);
          MmaFrags<Cfg> frags;
          mma_load<Cfg>(frags, tk, tv, m.nvalid, lane);
          mma_compute<Cfg>(state, frags, p, m, lane);
          if (issued < total) {
            produce<Cfg>(pr, p, &tmK, &tmV, tiles, meta, bars, stage, lane, &cta_flags);
            ++issued;
          }
        } else {
          if (m.flags & kFirst) simt_begin<Cfg>(state, p, m, qbuf, lane);
          simt_block<Cfg>(state, p, m, tk, tv, qbuf, lane);
          if (issued < total) {
            produce<Cfg>(pr, p, &tmK, &tmV, tiles, meta, bars, stage, lane, &cta_flags);
            ++issued;
          }
        }
        if (m.flags & kLast) {
          if constexpr (Cfg::MMA)
            mma_finish<Cfg>(state, p, m, w, lane);
          else
            simt_finish<Cfg>(state, p, m, w, lane);
        }
      }
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) p.cta_flags[blockIdx.x] = cta_flags;
  grid_dep_launch();
}

template <class Cfg>
DecodeKernel decode_entry() {
  DecodeKernel k;
  k.fn = reinterpret_cast<const void *>(&decode_kernel<Cfg>);
  k.mma = Cfg::MMA ? 1 : 0;
  k.cache_dtype = Cfg::Cache::kCode;
  k.q_dtype = Cfg::Q::kCode;
  k.D = Cfg::D;
  k.GC = Cfg::GC;
  k.warps = Cfg::WARPS;
  k.stages = Cfg::STAGES;
  k.smem_bytes = Cfg::SMEM;
  return k;
}

// Default pipeline shape: 5 warps per CTA, 16 KiB of stages per warp (two
// bf16 D=128 blocks), two CTAs per SM — the fastest of the shapes measured on
// GB300 for the GQA-8 layer (10 warps x 2 stages beat 8 x 3, 12 x 2 and 4 x 6).
constexpr int kWarps = 5;
constexpr int kBudget = 16 * 1024;  // shared-memory pipeline bytes per warp

}  // namespace pkv
