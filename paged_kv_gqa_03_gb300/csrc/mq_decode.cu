// mq_decode.cu — multi-query paged decode on the fifth-generation tensor cores
// with the score matrix transposed: q_len new tokens per sequence (a
// speculative-decoding verify step or a short chunk), token i attending the
// first ctx - (q_len - 1 - i) positions of its sequence's paged cache.
//
// What it computes is the attention of "LLM推理优化实战" §3.2 (flash_attention:
// K / V in blocks, online softmax with running max m and sum l, O rescaled by
// exp(m_old - m_new)) with the causal mask among new tokens of "苦猿的大模型
// 日记 Day45" PART 04, over the block table of "大模型推理加速——KV Cache篇"
// §6.1; partial results of one (sequence, kv head) split between CTAs are
// merged by their log-sum-exp (Flash-Decoding, "苦猿的大模型日记 Day45" PART 03).
//
// GB300 design.  A kv head serves only R = q_len * G <= 64 query rows, so a
// 128-row tile (M = 128 on the tensor core) would be mostly padding.  The
// positions take the M side instead:
//  * S^T = K . Q^T per tile of 128 positions: A = the K tile (K-major, as the
//    TMA lands it), B = Q (K-major, NR = 16 / 32 / 64 rows), D = 128 lanes
//    (positions) x NR columns (query rows) of tensor memory;
//  * softmax with one thread per (position, half of the rows): the row max of
//    a tile is a reduce-scatter over the warp's 32 positions plus an exchange
//    between the four warps of a half; the row sum stays per thread until an
//    item ends;
//  * O^T += V^T . P^T: A = the V tile read MN-major (the head dim contiguous),
//    B = P^T written by the softmax threads as one row of NR 16-bit values per
//    position (MN-major, the query rows contiguous; 32 / 64 / 128-byte
//    swizzle for NR = 16 / 32 / 64).  For a bf16 cache P
//    goes in as a bf16 high part plus its bf16 residual (two MMAs per k-step,
//    ~16 significant bits; bf16 alone gives 8, too few for the 2e-3 bound), so
//    V needs no conversion; an f16 cache takes f16 P directly;
//  * stream-K scheduling: the (sequence, kv head) items' K / V tiles form one
//    sequence that is cut into equal ranges, one per CTA (one CTA per SM); an
//    item cut by a range end is finished by the merge kernel from the CTAs'
//    normalised partial outputs and log-sum-exps;
//  * warp roles: 0-7 softmax / epilogue / Q staging, 8 and 11 TMA producers of
//    the K and the V tiles (block ids loaded three tiles ahead and first used
//    when the copies are issued), 9 S^T issue and tensor-memory allocation,
//    10 P . V issue.  Every wait is bounded; a timeout sets PKV_FLAG_TIMEOUT, and
//    the CTA drains its copies and MMAs and frees its tensor memory.
#include <math.h>

#include "mq_decode.h"
#include "prefill_common.cuh"

namespace pkv {

// T: the cache type; QT: the query / output type (= T for 16-bit caches).
// An fp8 cache is widened to f16 in shared memory (exact: every E4M3 value
// is an f16 value) and the MMAs run on f16 (Q converted when staged), so
// BF (the MMA operand type) is false for it while OUT_BF follows the query.
template <class T, int NRH_, class QT = T>
struct MqCfg {
  static constexpr int D = kMqHeadDim;
  static constexpr bool FP8 = T::kBytes == 1;
  static constexpr bool BF = !FP8 && T::kCode == PKV_BF16;
  static constexpr bool OUT_BF = QT::kCode == PKV_BF16;
  static constexpr int NRH = NRH_;                      // query rows of one softmax half
  static constexpr int NR = 2 * NRH;                    // S^T columns (rows padded)
  static constexpr int NPV = NR;                        // P^T columns (the padded rows)
  static constexpr int P_ROW = 2 * NR;                  // bytes of one position's P^T row: 32 / 64 / 128
  static constexpr uint32_t P_LAYOUT = NR == 16 ? 6u : (NR == 32 ? 4u : 2u);  // 32 / 64 / 128-byte swizzle
  static constexpr int N = 128;                         // positions per K / V tile
  static constexpr int BLOCKS = N / kBlock;             // paged blocks per tile
  static constexpr int PANELS = D / 64;                 // 128-byte panels per K / V row
  static constexpr int PANEL_KV = N * 128;
  static constexpr int KV_BYTES = PANELS * PANEL_KV;    // one K (or V) tile
  static constexpr int PANEL_Q = NR * 128;
  static constexpr int Q_BYTES = PANELS * PANEL_Q;
  static constexpr int PARTS = BF ? 2 : 1;              // P: bf16 high part + residual, or f16
  static constexpr int P_PART = N * P_ROW;
  static constexpr int P_BYTES = PARTS * P_PART;
  // rings as deep as shared memory allows: a V slot is held from its copy to
  // the end of its P . V, so V gets the depth.  fp8: the copies land in raw
  // rings of RAW_BYTES tiles (one 128-byte panel per position), the producers
  // widen each tile into the f16 operand rings below.
  // fp8: two raw slots per tensor; the softmax warps widen tile g + 1 while
  // they process tile g, into two-deep f16 rings
  static constexpr int KSTAGES = FP8 ? 2 : (NR <= 32 ? 3 : 2), VSTAGES = FP8 ? 2 : 3;
  static constexpr int PBUF = NR <= 16 ? 2 : 1, SBUF = 2;
  static constexpr int QBUF = NR <= 16 ? 2 : 1;
  static constexpr int RAW_BYTES = N * D;               // one fp8 K (or V) tile
  static constexpr int KRAW = FP8 ? 2 : 0, VRAW = FP8 ? 2 : 0;
  static constexpr int SC_RING = 8;                     // fp8 block scales of the tiles in flight
  static constexpr int LOADS = FP8 ? BLOCKS : BLOCKS * PANELS;  // TMA boxes per K (or V) tile
  static constexpr size_t SMEM = 1024 + (size_t)(KSTAGES + VSTAGES) * KV_BYTES + (size_t)PBUF * P_BYTES +
                                 (size_t)QBUF * Q_BYTES + (size_t)(KRAW + VRAW) * RAW_BYTES;
  // 16-byte chunk c of position kt's P^T row, swizzled as the P . V operand reads it
  __device__ static __forceinline__ int p_chunk(int kt, int c) {
    return c ^ (NR == 16 ? (kt >> 2) & 1 : (NR == 32 ? (kt >> 1) & 3 : kt & 7));
  }
  static constexpr uint32_t COL_O = 128;                // two O^T buffers of NPV columns after the S^T buffers
  static constexpr uint32_t TMEM_COLS = 256;
  static constexpr int SOFTMAX = 256;                   // 128 positions x 2 halves of the rows
  static constexpr int THREADS = SOFTMAX + 128;        // + K producer, S^T issuer, P . V issuer, V producer
  static constexpr int PRODUCER = SOFTMAX / 32, ISSUER = PRODUCER + 1, PV_ISSUER = PRODUCER + 2,
                       V_PRODUCER = PRODUCER + 3;
  static_assert(NRH == 8 || NRH == 16 || NRH == 32, "rows per half");
  static_assert(!FP8 || NRH <= 16, "fp8: up to 32 rows (shared memory)");
  static_assert(SBUF * NR <= (int)COL_O && COL_O + 2 * NPV <= TMEM_COLS, "tensor memory");
  static_assert(LOADS <= 32, "one box per producer lane");
  static_assert(SMEM + 4096 <= 232448, "shared memory");
};

// Warp reduce-scatter of NRH values per lane: afterwards lane l holds the
// maximum (or sum) over the warp's 32 lanes of value l % NRH.  Steps of
// distance >= NRH exchange every value; the later ones halve the set, lanes
// with the distance bit set keeping the upper half.
template <int NRH, bool MAX>
__device__ __forceinline__ float reduce_scatter(float (&v)[NRH], int lane) {
#pragma unroll
  for (int k = 16; k >= NRH; k >>= 1)
#pragma unroll
    for (int e = 0; e < NRH; ++e) {
      const float o = __shfl_xor_sync(kFull, v[e], k);
      v[e] = MAX ? fmaxf(v[e], o) : v[e] + o;
    }
#pragma unroll
  for (int n = NRH; n > 1; n >>= 1) {
    const int k = n >> 1;
    const bool up = (lane & k) != 0;
#pragma unroll
    for (int e = 0; e < k; ++e) {
      const float send = up ? v[e] : v[e + k];
      const float keep = up ? v[e + k] : v[e];
      const float o = __shfl_xor_sync(kFull, send, k);
      v[e] = MAX ? fmaxf(keep, o) : keep + o;
    }
  }
  return v[0];
}

// Tile facts of one sequence: the clamped context, the first position any
// new token's window reaches, the first K / V tile and the tile count T (per
// kv head).  Token i sees positions [ctx - q_len + 1 + i - window, ctx - q_len
// + 1 + i) (no lower bound without a window).
struct MqSeq {
  int ctx, first, j_first, T;
  bool bad_ctx;
};
__device__ __forceinline__ MqSeq mq_seq(const MqParams &p, int b) {
  MqSeq s;
  const int raw = __ldg(p.context_lens + b);
  const int cap = p.max_blocks * kBlock;
  s.ctx = raw < 0 ? 0 : (raw > cap ? cap : raw);
  s.bad_ctx = raw != s.ctx;
  const int lim_lo = s.ctx - p.q_len + 1;  // exclusive end of token 0's positions
  s.first = p.window > 0 ? max(0, lim_lo - p.window) : 0;
  s.j_first = s.first / 128;
  s.T = s.ctx > 0 ? (s.ctx - 1) / 128 - s.j_first + 1 : 0;
  return s;
}

// A CTA's share of the stream-K order: tiles [t0, t1) of the sequence of all
// items' tiles (item (b, h) holds tiles [prefix[b] + h * T_b, ... + T_b)).
// One segment = the part of one item inside the range; every role walks the
// same segments.
struct MqSeg {
  int b, h, j0, j1, T, ctx, first, j_first;
  int slot;    // partial-output slot of a cut item: 0 if the segment starts the CTA's range, else 1
  bool whole;  // the segment is the whole item (the CTA writes the output itself)
};
struct MqWalk {
  int t, t0, t1, b, base;  // next tile; the range; the sequence holding tile t and its first tile
  __device__ __forceinline__ void start(int b0, int base0, int tile0, int tile1) {
    b = b0;
    base = base0;
    t = t0 = tile0;
    t1 = tile1;
  }
  __device__ __forceinline__ bool next(const MqParams &p, MqSeg &sg) {
    if (t >= t1) return false;
    MqSeq s = mq_seq(p, b);
    while (t >= base + s.T * p.Hkv) {  // on to the sequence holding tile t (skipping empty ones)
      base += s.T * p.Hkv;
      s = mq_seq(p, ++b);
    }
    const int off = t - base;
    sg.b = b;
    sg.T = s.T;
    sg.h = off / s.T;
    sg.j0 = off - sg.h * s.T;
    sg.j1 = min(s.T, sg.j0 + (t1 - t));
    sg.ctx = s.ctx;
    sg.first = s.first;
    sg.j_first = s.j_first;
    sg.slot = t == t0 ? 0 : 1;
    sg.whole = sg.j0 == 0 && sg.j1 == s.T;
    t += sg.j1 - sg.j0;
    return true;
  }
};

// S^T = K . Q^T of one tile into tensor-memory columns dS (128 lanes =
// positions, NR columns = query rows): D / 16 MMAs over the K tile (A,
// K-major, at k0) and Q (B, K-major, NR rows, at q0).  Issued by one thread.
template <class Cfg>
__device__ __forceinline__ void mma_st_tile(uint32_t dS, uint32_t k0, uint32_t q0) {
  constexpr uint32_t id = tc::idesc_f16_ab(Cfg::BF, 128, Cfg::NR, false, false);
#pragma unroll
  for (int k = 0; k < Cfg::D / 16; ++k) {
    const uint32_t offk = (uint32_t)((k >> 2) * Cfg::PANEL_KV + (k & 3) * 32);
    const uint32_t offq = (uint32_t)((k >> 2) * Cfg::PANEL_Q + (k & 3) * 32);
    tc::mma_f16(dS, tc::desc_sw128(k0 + offk, 16, 1024), tc::desc_sw128(q0 + offq, 16, 1024), id, k > 0 ? 1u : 0u);
  }
}

// O^T (+)= V^T . P^T of one tile into dO (128 lanes = head dim, NPV columns
// = query rows): A = the V tile read MN-major (the head dim contiguous, two
// 64-element panels), B = each P part (MN-major, one P_ROW-byte row per
// position); 16 positions per MMA.  `accumulate` false starts O^T afresh.
template <class Cfg>
__device__ __forceinline__ void mma_pvt_tile(uint32_t dO, uint32_t v0, uint32_t p0, bool accumulate) {
  constexpr uint32_t id = tc::idesc_f16_ab(Cfg::BF, 128, Cfg::NPV, true, true);
#pragma unroll
  for (int k = 0; k < Cfg::N / 16; ++k) {
    const uint64_t dv = tc::desc_sw128(v0 + (uint32_t)k * 2048, Cfg::PANEL_KV, 1024);
#pragma unroll
    for (int part = 0; part < Cfg::PARTS; ++part) {
      // 16 positions = 16 P^T rows; 8-row swizzle atoms P_ROW * 8 bytes apart
      const uint64_t dp = tc::desc_sw(p0 + (uint32_t)(part * Cfg::P_PART + k * 16 * Cfg::P_ROW), Cfg::P_PART,
                                      8 * Cfg::P_ROW, Cfg::P_LAYOUT);
      tc::mma_f16(dO, dv, dp, id, (accumulate || k > 0 || part > 0) ? 1u : 0u);
    }
  }
}

// Warp-wide load of NRH consecutive tensor-memory columns of the warp's 32
// lanes (with its wait).
template <int NRH>
__device__ __forceinline__ void ld_cols(uint32_t ta, uint32_t (&r)[NRH]) {
  if constexpr (NRH == 8)
    tc::ld8(ta, r);
  else if constexpr (NRH == 16)
    tc::ld16(ta, r);
  else
    tc::ld32(ta, r);
}

// fp8 caches: the softmax threads' widening of one landed E4M3 tile (TMA
// layout: 128 rows of 128 bytes, 128-byte swizzle) into the f16 operand
// layout of a 16-bit tile (two 64-element panels of 128-byte rows, 128-byte
// swizzle), the layout the MMAs read K (K-major) and V (MN-major) from.  Each
// E4M3 value is an f16 value, so the widening is exact; rows at or past
// zero_from (stale positions past the context) become zeros.  Thread t takes
// the 16-byte chunks t, t + 256, t + 512, t + 768 (eight threads per row:
// conflict-free loads), its four loads in flight together.
template <class Cfg>
__device__ __forceinline__ void widen_share(const uint8_t *raw, uint8_t *op, int zero_from, int tid) {
  constexpr int PER = Cfg::N * 8 / Cfg::SOFTMAX;  // chunks of a thread
  const uint32_t rb = smem_u32(raw), ob = smem_u32(op);
  uint4 x[PER];
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int i = tid + k * Cfg::SOFTMAX, r = i >> 3, c = i & 7;
    x[k] = lds128(rb + (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)));
  }
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int i = tid + k * Cfg::SOFTMAX, r = i >> 3, c = i & 7;
    uint4 lo = make_uint4(0, 0, 0, 0), hi = make_uint4(0, 0, 0, 0);
    if (r < zero_from) {
      lo = make_uint4(e4m3x2_to_f16x2((uint16_t)(x[k].x & 0xffff)), e4m3x2_to_f16x2((uint16_t)(x[k].x >> 16)),
                      e4m3x2_to_f16x2((uint16_t)(x[k].y & 0xffff)), e4m3x2_to_f16x2((uint16_t)(x[k].y >> 16)));
      hi = make_uint4(e4m3x2_to_f16x2((uint16_t)(x[k].z & 0xffff)), e4m3x2_to_f16x2((uint16_t)(x[k].z >> 16)),
                      e4m3x2_to_f16x2((uint16_t)(x[k].w & 0xffff)), e4m3x2_to_f16x2((uint16_t)(x[k].w >> 16)));
    }
    // elements 16c .. 16c + 15: panel c / 4, 16-byte chunks 2 (c % 4) and
    // 2 (c % 4) + 1.  The two panels share banks, so threads of panel 1 store
    // their odd chunk first: each store's eight threads of a row then cover
    // all 32 banks (no conflict)
    const uint32_t row = ob + (uint32_t)((c >> 2) * Cfg::PANEL_KV + r * 128);
    const int ch = (c & 3) * 2;
    const bool odd_first = c >= 4;
    sts128(row + (uint32_t)(((ch + (odd_first ? 1 : 0)) ^ (r & 7)) << 4), odd_first ? hi : lo);
    sts128(row + (uint32_t)(((ch + (odd_first ? 0 : 1)) ^ (r & 7)) << 4), odd_first ? lo : hi);
  }
}

// A query row (16-byte chunk of 8 values) as the MMA operand type: f16 for
// fp8 caches (a bf16 query converted, exact for normal f16 magnitudes),
// unchanged otherwise.
template <class Cfg>
__device__ __forceinline__ uint4 q_chunk(uint4 v) {
  if constexpr (Cfg::FP8 && Cfg::OUT_BF) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t h[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) h[e] = pack_f16x2(__uint_as_float(w[e] << 16), __uint_as_float(w[e] & 0xffff0000u));
    return make_uint4(h[0], h[1], h[2], h[3]);
  } else {
    return v;
  }
}

template <class Cfg>
__global__ void __launch_bounds__(Cfg::THREADS, 1)
    mq_decode_kernel(const __grid_constant__ MqParams p, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV) {
  constexpr int NRH = Cfg::NRH, NR = Cfg::NR;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t *sK = smem;
  uint8_t *sV = sK + (size_t)Cfg::KSTAGES * Cfg::KV_BYTES;
  uint8_t *sP = sV + (size_t)Cfg::VSTAGES * Cfg::KV_BYTES;
  uint8_t *sQ = sP + (size_t)Cfg::PBUF * Cfg::P_BYTES;
  uint8_t *sKr = sQ + (size_t)Cfg::QBUF * Cfg::Q_BYTES;     // fp8: raw K / V rings
  uint8_t *sVr = sKr + (size_t)Cfg::KRAW * Cfg::RAW_BYTES;
  __shared__ __align__(8) uint64_t k_full[Cfg::KSTAGES], k_empty[Cfg::KSTAGES];
  // fp8: raw K / V tiles landed / widened (the widened tiles are announced on k_full / v_full)
  __shared__ __align__(8) uint64_t kr_full[Cfg::FP8 ? Cfg::KRAW : 1], vr_full[Cfg::FP8 ? Cfg::VRAW : 1];
  __shared__ __align__(8) uint64_t kr_empty[Cfg::FP8 ? Cfg::KRAW : 1], vr_empty[Cfg::FP8 ? Cfg::VRAW : 1];
  __shared__ int raw_zero[Cfg::FP8 ? Cfg::VRAW : 1];        // fp8 V: first stale row of each raw tile
  __shared__ int kr_issued, vr_issued;                      // fp8: raw copies issued
  __shared__ __align__(8) uint64_t v_full[Cfg::VSTAGES], v_empty[Cfg::VSTAGES];
  // S^T landed / read out of tensor memory; P written / P . V done (P buffer free)
  __shared__ __align__(8) uint64_t s_full[Cfg::SBUF], s_free[Cfg::SBUF], p_full[Cfg::PBUF], pv_done[Cfg::PBUF];
  // per segment: Q staged, O^T read out; row-max exchange per tile, row-sum exchange per segment
  __shared__ __align__(8) uint64_t q_full[Cfg::QBUF], o_free[2], xch[2][2], xl[2], fin;
  __shared__ float red[2][2][4][32];  // partial row maxima [tile parity][half][warp quarter][row]
  __shared__ float red_l[2][4][32];   // partial row sums [half][warp quarter][row]
  __shared__ int32_t s_wsum[8], s_b0, s_base0;  // per-warp tile sums; where the CTA's range starts
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag, cta_flags, k_consumed, v_consumed, k_issued, v_issued;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < Cfg::KSTAGES; ++s) {
      mbar_init(&k_full[s], Cfg::FP8 ? Cfg::SOFTMAX / 32 : 1);  // fp8: every softmax warp's share widened
      mbar_init(&k_empty[s], 1);
    }
#pragma unroll
    for (int s = 0; s < Cfg::VSTAGES; ++s) {
      mbar_init(&v_full[s], Cfg::FP8 ? Cfg::SOFTMAX / 32 : 1);
      mbar_init(&v_empty[s], 1);
    }
#pragma unroll
    for (int s = 0; s < Cfg::SBUF; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&s_free[s], Cfg::SOFTMAX / 32);
    }
#pragma unroll
    for (int s = 0; s < Cfg::PBUF; ++s) {
      mbar_init(&p_full[s], Cfg::SOFTMAX / 32);
      mbar_init(&pv_done[s], 1);
    }
#pragma unroll
    for (int s = 0; s < Cfg::QBUF; ++s) mbar_init(&q_full[s], Cfg::SOFTMAX / 32);
    mbar_init(&o_free[0], Cfg::SOFTMAX / 32);
    mbar_init(&o_free[1], Cfg::SOFTMAX / 32);
    mbar_init(&xch[0][0], 4);
    mbar_init(&xch[0][1], 4);
    mbar_init(&xch[1][0], 4);
    mbar_init(&xch[1][1], 4);
    mbar_init(&xl[0], 4);
    mbar_init(&xl[1], 4);
    mbar_init(&fin, 2);  // one commit from each issuing warp
    if constexpr (Cfg::FP8) {
#pragma unroll
      for (int s = 0; s < Cfg::KRAW; ++s) {
        mbar_init(&kr_full[s], 1);
        mbar_init(&kr_empty[s], Cfg::SOFTMAX / 32);
      }
#pragma unroll
      for (int s = 0; s < Cfg::VRAW; ++s) {
        mbar_init(&vr_full[s], 1);
        mbar_init(&vr_empty[s], Cfg::SOFTMAX / 32);
      }
    }
    fence_barrier_init();
    abort_flag = 0;
    cta_flags = 0;
    k_consumed = v_consumed = k_issued = v_issued = 0;
    kr_issued = vr_issued = 0;
  }
  if (warp == Cfg::ISSUER) tc::alloc(&tmem_base, Cfg::TMEM_COLS);
  if (warp == Cfg::PRODUCER && lane == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  // launched early behind the previous kernel: its writes (the appended
  // tokens, the step's bookkeeping) are visible from here on
  grid_dep_wait();
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tbase = tmem_base;

  // ---- tile prefix over the sequences (256 threads, up to 8 sequences each):
  // the total, where this CTA's range starts, and (CTA 0) the prefix for the
  // merge kernel ----
  const int B = p.B;
  const int per = (B + Cfg::SOFTMAX - 1) / Cfg::SOFTMAX;
  int tk[kMqMaxBatch / Cfg::SOFTMAX];
  int own = 0, incl = 0;
  if (tid < Cfg::SOFTMAX) {
    int bad = 0;
#pragma unroll
    for (int k = 0; k < kMqMaxBatch / Cfg::SOFTMAX; ++k) {
      const int b = tid * per + k;
      tk[k] = 0;
      if (k < per && b < B) {
        const MqSeq s = mq_seq(p, b);
        tk[k] = s.T * p.Hkv;
        bad |= s.bad_ctx ? 1 : 0;
      }
      own += tk[k];
    }
    incl = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += n;
    }
    if (lane == 31) s_wsum[warp] = incl;
    if (blockIdx.x == 0 && __any_sync(kFull, bad) && lane == 0) atomicOr(&cta_flags, PKV_FLAG_BAD_LEN);
  }
  __syncthreads();
  int W = 0;
#pragma unroll
  for (int w = 0; w < Cfg::SOFTMAX / 32; ++w) W += s_wsum[w];
  const int t0 = (int)((int64_t)W * blockIdx.x / gridDim.x);
  const int t1 = (int)((int64_t)W * (blockIdx.x + 1) / gridDim.x);
  if (tid == 0) {  // an empty range (t0 == W): nothing to walk
    s_b0 = B;
    s_base0 = W;
    if (blockIdx.x == 0) p.prefix[B] = W;
  }
  __syncthreads();
  if (tid < Cfg::SOFTMAX) {
    int run = incl - own;
    for (int w = 0; w < warp; ++w) run += s_wsum[w];
#pragma unroll
    for (int k = 0; k < kMqMaxBatch / Cfg::SOFTMAX; ++k) {
      const int b = tid * per + k;
      if (k < per && b < B) {
        if (blockIdx.x == 0) p.prefix[b] = run;
        if (run <= t0 && t0 < run + tk[k]) {  // the sequence holding the range's first tile
          s_b0 = b;
          s_base0 = run;
        }
        run += tk[k];
      }
    }
  }
  __syncthreads();
  const int b0 = s_b0, base0 = s_base0;

  if (warp == Cfg::PRODUCER || warp == Cfg::V_PRODUCER) {
    // ---------------- TMA producers: K tiles (warp 8), V tiles (warp 11) ----------------
    // two warps, so neither tensor's copies wait behind the other's issue;
    // lane l fetches block (l % 8) of a tile, panel l / 8; a cursor walks the
    // CTA's tiles, fetching block ids three tiles ahead
    const int slot = lane & (Cfg::BLOCKS - 1), panel = lane / Cfg::BLOCKS;
    MqWalk wk;
    wk.start(b0, base0, t0, t1);
    MqSeg cs{};
    int cj = 0;
    bool have = false;
    auto step = [&]() -> bool {  // to the cursor's next tile; false past the CTA's last
      if (have && ++cj < cs.j1) return true;
      have = wk.next(p, cs);
      if (have) cj = cs.j0;
      return have;
    };
    int bad = 0;
    // this lane's block of the cursor tile: its raw id, loaded here and first
    // used when the tile's copies are issued (three tiles on), so the load's
    // latency is hidden; none = past the context, or wholly before every new
    // token's window (such blocks may have been released)
    struct Pend {
      int id, h;
      bool none;
      int zf;  // fp8 V: the tile's first row past the context (zeroed when widened)
    };
    auto fetch = [&]() -> Pend {
      Pend f;
      const int lb = (cs.j_first + cj) * Cfg::BLOCKS + slot;
      const int nblk = (cs.ctx + kBlock - 1) / kBlock;
      f.h = cs.h;
      f.none = lb >= nblk || (lb + 1) * kBlock <= cs.first;
      f.id = f.none ? 0 : __ldg(p.block_table + (size_t)cs.b * p.max_blocks + lb);
      f.zf = cs.ctx - (cs.j_first + cj) * Cfg::N;
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
    const Pend nil{0, 0, true, 0};
    bool h0 = step();
    Pend f0 = h0 ? fetch() : nil;
    bool h1 = h0 && step();
    Pend f1 = h1 ? fetch() : nil;
    bool h2 = h1 && step();
    Pend f2 = h2 ? fetch() : nil;
    if constexpr (Cfg::FP8) {
      // fp8: the tiles land raw (RAW ring); the softmax warps widen tile g + 1
      // into the f16 operand ring while they process tile g and then release
      // its raw slot (kr_empty / vr_empty), which this warp reissues
      static_assert(Cfg::KRAW == Cfg::VRAW, "same raw ring depths for K and V");
      constexpr int RAWN = Cfg::KRAW;
      uint8_t *raw = vw ? sVr : sKr;
      uint64_t *rbar = vw ? vr_full : kr_full;
      uint64_t *rfree = vw ? vr_empty : kr_empty;
      const CUtensorMap *tm = vw ? &tmV : &tmK;
      int *r_issued = vw ? &vr_issued : &kr_issued;
      for (int g = 0; h0 && ok; ++g) {
        const bool h3 = h2 && step();
        const Pend f3 = h3 ? fetch() : nil;
        const int rs = g % RAWN;
        if (g >= RAWN) ok = warp_wait(&rfree[rs], (uint32_t)((g / RAWN) - 1) & 1u, p.timeout_ns);
        if (ok && __any_sync(kFull, *(volatile int *)&abort_flag)) ok = false;
        if (!ok) break;
        const int64_t trow = row_of(f0);
        if (lane == 0) {
          if (vw) raw_zero[rs] = f0.zf;
          mbar_arrive_expect_tx(&rbar[rs], Cfg::RAW_BYTES);
        }
        __syncwarp();
        if (lane < Cfg::LOADS)
          tma_load_2d(raw + (size_t)rs * Cfg::RAW_BYTES + slot * 2048, tm, 0, (int)(trow * kBlock), &rbar[rs]);
        if (lane == 0) *r_issued = g + 1;
        h0 = h1;
        f0 = f1;
        h1 = h2;
        f1 = f2;
        h2 = h3;
        f2 = f3;
      }
    } else {
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
    }
    if (__any_sync(kFull, bad) && lane == 0) atomicOr(&cta_flags, PKV_FLAG_BAD_BLOCK);
    if (!ok && lane == 0) {
      atomicOr(&cta_flags, PKV_FLAG_TIMEOUT);
      abort_flag = 1;
    }
  } else if (warp == Cfg::ISSUER) {
    // ---------------- S^T issue ----------------
    // in tile order as K lands; a segment's first S^T waits for its Q.  (P . V
    // has a warp of its own: the two write different tensor-memory columns
    // and read different shared memory, so neither waits behind the other's
    // inputs; each warp's commits track its own MMAs.)
    bool ok = true;
    MqWalk wk;
    wk.start(b0, base0, t0, t1);
    MqSeg sg{};
    int g = 0;
    for (int si = 0; ok && wk.next(p, sg); ++si) {
      const int qb = si % Cfg::QBUF;
      ok = warp_wait(&q_full[qb], (uint32_t)(si / Cfg::QBUF) & 1u, p.timeout_ns);
      for (int j = sg.j0; ok && j < sg.j1; ++j, ++g) {
        const int ks = g % Cfg::KSTAGES, sb = g % Cfg::SBUF;
        ok = warp_wait(&k_full[ks], (uint32_t)(g / Cfg::KSTAGES) & 1u, p.timeout_ns);
        if (ok && g >= Cfg::SBUF) ok = warp_wait(&s_free[sb], (uint32_t)((g / Cfg::SBUF) - 1) & 1u, p.timeout_ns);
        if (!ok) break;
        if (lane == 0) k_consumed = g + 1;
        tc::fence_after();
        if (lane == 0) {
          mma_st_tile<Cfg>(tbase + (uint32_t)(sb * NR), smem_u32(sK + (size_t)ks * Cfg::KV_BYTES),
                           smem_u32(sQ + (size_t)qb * Cfg::Q_BYTES));
          tc::commit(&s_full[sb]);
          tc::commit(&k_empty[ks]);
        }
        __syncwarp();
        if (__any_sync(kFull, *(volatile int *)&abort_flag)) ok = false;
      }
    }
    if (!ok && lane == 0) {
      atomicOr(&cta_flags, PKV_FLAG_TIMEOUT);
      abort_flag = 1;
    }
  } else if (warp == Cfg::PV_ISSUER) {
    // ---------------- P . V issue ----------------
    // in tile order once V has landed and P is written; a segment's first
    // P . V waits for the O^T buffer it reuses (read out two segments ago)
    bool ok = true;
    MqWalk wk;
    wk.start(b0, base0, t0, t1);
    MqSeg sg{};
    int g = 0;
    for (int si = 0; ok && wk.next(p, sg); ++si) {
      const int ob = si & 1;
      if (si >= 2) ok = warp_wait(&o_free[ob], (uint32_t)((si >> 1) - 1) & 1u, p.timeout_ns);
      const int nblk = (sg.ctx + kBlock - 1) / kBlock;
      for (int j = sg.j0; ok && j < sg.j1; ++j, ++g) {
        const int vs = g % Cfg::VSTAGES, pb = g % Cfg::PBUF;
        ok = warp_wait(&v_full[vs], (uint32_t)(g / Cfg::VSTAGES) & 1u, p.timeout_ns);
        if (ok) ok = warp_wait(&p_full[pb], (uint32_t)(g / Cfg::PBUF) & 1u, p.timeout_ns);
        if (!ok) break;
        if (lane == 0) v_consumed = g + 1;
        uint8_t *vt = sV + (size_t)vs * Cfg::KV_BYTES;
        const int kv0 = (sg.j_first + j) * Cfg::N;  // first position of the tile
        if constexpr (!Cfg::FP8)  // (fp8: the widening wrote zeros there)
          zero_v_rows<Cfg>(vt, sg.ctx - kv0, min(nblk * kBlock - kv0, Cfg::N), lane);
        __syncwarp();
        tc::fence_after();
        if (lane == 0) {
          mma_pvt_tile<Cfg>(tbase + Cfg::COL_O + (uint32_t)(ob * Cfg::NPV), smem_u32(vt),
                            smem_u32(sP + (size_t)pb * Cfg::P_BYTES), j > sg.j0);
          tc::commit(&pv_done[pb]);
          tc::commit(&v_empty[vs]);
        }
        __syncwarp();
        if (__any_sync(kFull, *(volatile int *)&abort_flag)) ok = false;
      }
    }
    if (!ok && lane == 0) {
      atomicOr(&cta_flags, PKV_FLAG_TIMEOUT);
      abort_flag = 1;
    }
  } else {
    // ---------------- softmax + epilogue: thread (position, half of the rows) ----------------
    const int qd = warp & 3, hf = warp >> 2;
    const int kt = qd * 32 + lane;  // position in the tile = tensor-memory lane (and head dim in O^T)
    const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
    const int row0 = hf * NRH;      // this half's first query row
    const int rr = lane & (NRH - 1);
    const float c = p.scale_log2;
    // Q of segment s into buffer qb: NR rows x 16 chunks of 16 bytes, row r =
    // (new token r / G, query head r % G of kv head s.h), zeros past R
    auto stage_q = [&](const MqSeg &s, int qb, bool async) {
      uint8_t *q0 = sQ + (size_t)qb * Cfg::Q_BYTES;
      for (int i = tid; i < NR * 16; i += Cfg::SOFTMAX) {
        const int r = i >> 4, cc = i & 15;
        const uint32_t dst = smem_u32(q0 + (cc >> 3) * Cfg::PANEL_Q + r * 128 + (((cc & 7) ^ (r & 7)) << 4));
        if (r < p.R) {
          const int ii = r / p.G, gq = r - ii * p.G;
          const uint4 *src = reinterpret_cast<const uint4 *>(
              static_cast<const uint16_t *>(p.q) + (((size_t)s.b * p.q_len + ii) * p.Hq + s.h * p.G + gq) * Cfg::D) + cc;
          if (async && !Cfg::FP8)  // (fp8: Q is converted to f16 on the way, synchronously)
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
          else
            sts128(dst, q_chunk<Cfg>(__ldg(src)));
        } else {
          sts128(dst, make_uint4(0, 0, 0, 0));
        }
      }
    };
    auto release_q = [&](int qb, bool async) {
      if (async) asm volatile("cp.async.wait_all;" ::: "memory");
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(&q_full[qb]);
    };
    // fp8: widen K (or V) of the CTA's tile gt (its global index in the
    // walk) from its raw slot into the f16 ring, then announce it and free
    // the raw slot.  The ring slot is free: K(gt - 2)'s S has completed and
    // V(gt - 2)'s P . V has been waited for by the caller.
    const int ntiles = t1 - t0;
    auto widen = [&](int gt, bool v) -> bool {
      constexpr int RAWN = Cfg::KRAW > 0 ? Cfg::KRAW : 1;  // (16-bit caches never call this)
      const int rs = gt % RAWN, os = gt % Cfg::KSTAGES;
      if (!warp_wait(v ? &vr_full[rs] : &kr_full[rs], (uint32_t)(gt / RAWN) & 1u, p.timeout_ns)) return false;
      widen_share<Cfg>((v ? sVr : sKr) + (size_t)rs * Cfg::RAW_BYTES, (v ? sV : sK) + (size_t)os * Cfg::KV_BYTES,
                       v ? raw_zero[rs] : Cfg::N, tid);
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(v ? &v_full[os] : &k_full[os]);
        mbar_arrive(v ? &vr_empty[rs] : &kr_empty[rs]);
      }
      return true;
    };
    MqWalk wk;
    wk.start(b0, base0, t0, t1);
    MqSeg sg{}, nx{};
    bool have = wk.next(p, sg);
    bool nhave = have && wk.next(p, nx);
    if (have) {
      stage_q(sg, 0, false);
      release_q(0, false);
    }
    bool ok = true;
    if constexpr (Cfg::FP8) {  // the first tile's K and V
      if (ntiles > 0) ok = widen(0, false) && widen(0, true);
    }
    int g = 0, si = 0;
    float m_run[NRH], l_part[NRH];
    while (have && ok) {
      const int n = sg.j1 - sg.j0, ob = si & 1;
      // the next segment's Q: with two buffers its copy starts now (the
      // buffer's last reader, S^T of segment si - 1, has completed), with one
      // at this segment's last tile (once its last S^T has landed)
      bool staged = false;
      if (Cfg::QBUF == 2 && nhave) {
        stage_q(nx, (si + 1) % Cfg::QBUF, true);
        staged = true;
      }
#pragma unroll
      for (int e = 0; e < NRH; ++e) {
        m_run[e] = -INFINITY;
        l_part[e] = 0.f;
      }
      // fp8: the K and V scales of this position's block, software-pipelined
      // within the segment: the block id two tiles ahead and the scales one
      // tile ahead are loaded while this tile is processed (0 for positions
      // no block holds: masked anyway)
      const int nblk_s = (sg.ctx + kBlock - 1) / kBlock;
      auto block_id = [&](int jj) -> int {  // -1: no block / none to read
        const int lb = ((sg.j_first + sg.j0 + jj) * Cfg::N + kt) / kBlock;
        if (jj >= n || lb >= nblk_s || (lb + 1) * kBlock <= sg.first) return -1;
        return __ldg(p.block_table + (size_t)sg.b * p.max_blocks + lb);
      };
      auto scale_of = [&](int id, const float *tab) -> float {
        return id >= 0 && (int64_t)id < p.num_blocks ? __ldg(tab + (size_t)id * p.Hkv + sg.h) : 0.f;
      };
      [[maybe_unused]] float ksc_n = 0.f, vsc_n = 0.f;
      [[maybe_unused]] int id_nn = -1;
      if constexpr (Cfg::FP8) {
        const int id0 = block_id(0);
        ksc_n = scale_of(id0, p.k_scale);
        vsc_n = scale_of(id0, p.v_scale);
        id_nn = block_id(1);
      }
      for (int j = 0; j < n; ++j) {
        const int gj = g + j, sb = gj % Cfg::SBUF, par = gj & 1;
        const int pos = (sg.j_first + sg.j0 + j) * Cfg::N + kt;
        float ksc = 1.f, vsc = 1.f;
        if constexpr (Cfg::FP8) {
          ksc = ksc_n;
          vsc = vsc_n;
          ksc_n = scale_of(id_nn, p.k_scale);  // tile j + 1
          vsc_n = scale_of(id_nn, p.v_scale);
          id_nn = block_id(j + 2);
          // K of the next tile, so its S can run while this tile's softmax does
          if (gj + 1 < ntiles && !(ok = widen(gj + 1, false))) break;
        }
        ok = warp_wait(&s_full[sb], (uint32_t)(gj / Cfg::SBUF) & 1u, p.timeout_ns);
        if (!ok) break;
        tc::fence_after();
        // S^T of this thread's position and rows, masked: new token i sees the
        // position iff imin <= i < imin + window (imin = pos - ctx + q_len)
        const uint32_t scol = tbase + lane_base + (uint32_t)(sb * NR + row0);
        const int imin = pos - sg.ctx + p.q_len;
        const int rlo = imin > 0 ? (imin < p.q_len ? imin * p.G : p.R) : 0;
        const int rhi = p.window > 0 ? (imin + p.window >= p.q_len ? p.R : max(0, imin + p.window) * p.G) : p.R;
        float s[NRH];
        auto load_s = [&]() {
          uint32_t sr[NRH];
          ld_cols<NRH>(scol, sr);
#pragma unroll
          for (int e = 0; e < NRH; ++e) s[e] = __uint_as_float(sr[e]) * ksc;  // (fp8: the block's K scale)
          if (!(rlo <= row0 && rhi >= row0 + NRH)) {
#pragma unroll
            for (int e = 0; e < NRH; ++e)
              if (row0 + e < rlo || row0 + e >= rhi) s[e] = -INFINITY;
          }
        };
        auto release_s = [&]() {
          tc::fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&s_free[sb]);
        };
        load_s();
        // the tile's row maxima over all 128 positions (with 32 rows a half
        // the reduction consumes s, which is loaded again afterwards:
        // registers)
        float mrow;
        if constexpr (NRH == 32) {
          mrow = reduce_scatter<NRH, true>(s, lane);
        } else {
          release_s();
          float mx[NRH];
#pragma unroll
          for (int e = 0; e < NRH; ++e) mx[e] = s[e];
          mrow = reduce_scatter<NRH, true>(mx, lane);
        }
        if (Cfg::QBUF == 1 && j + 1 == n && nhave) {
          stage_q(nx, 0, true);
          staged = true;
        }
        if (lane < NRH) red[par][hf][qd][lane] = mrow;
        __syncwarp();
        if (lane == 0) mbar_arrive(&xch[par][hf]);
        ok = warp_wait(&xch[par][hf], (uint32_t)(gj >> 1) & 1u, p.timeout_ns);
        if (!ok) break;
        if constexpr (NRH == 32) {
          load_s();
          release_s();
        }
        const float mt = fmaxf(fmaxf(red[par][hf][0][rr], red[par][hf][1][rr]),
                               fmaxf(red[par][hf][2][rr], red[par][hf][3][rr]));
        // running maxima move only when a row's grows by more than 2^8: P and l
        // share the stale max, so the result is exact either way
        bool need = false;
#pragma unroll
        for (int e = 0; e < NRH; ++e) need |= fmaxf(m_run[e], __shfl_sync(kFull, mt, e) * c) > m_run[e] + 8.f;
        if (__any_sync(kFull, need)) {
          // O^T holds this segment's earlier tiles (j > 0): P . V(gj - 1) must be
          // done before it is scaled, and P . V(gj) is issued after the arrival
          // below; 8 rows at a time (registers)
          if (j > 0) {
            const int gp = gj - 1;
            ok = warp_wait(&pv_done[gp % Cfg::PBUF], (uint32_t)(gp / Cfg::PBUF) & 1u, p.timeout_ns);
            if (!ok) break;
            tc::fence_after();
          }
          const uint32_t ta = tbase + lane_base + Cfg::COL_O + (uint32_t)(ob * Cfg::NPV + row0);
#pragma unroll
          for (int k = 0; k < NRH / 8; ++k) {
            float alpha[8];
#pragma unroll
            for (int e8 = 0; e8 < 8; ++e8) {
              const int e = 8 * k + e8;
              const float mn = fmaxf(m_run[e], __shfl_sync(kFull, mt, e) * c);
              alpha[e8] = 1.f;
              if (mn > m_run[e] + 8.f) {
                alpha[e8] = ex2(m_run[e] - mn);
                m_run[e] = mn;
                l_part[e] *= alpha[e8];
              }
            }
            if (j > 0) {
              uint32_t o[8];
              tc::ld8(ta + (uint32_t)(8 * k), o);
#pragma unroll
              for (int e8 = 0; e8 < 8; ++e8) o[e8] = __float_as_uint(__uint_as_float(o[e8]) * alpha[e8]);
              tc::st8(ta + (uint32_t)(8 * k), o[0], o[1], o[2], o[3], o[4], o[5], o[6], o[7]);
            }
          }
          if (j > 0) tc::wait_st();
        }
        // P (in place of S) and the per-thread row sums
#pragma unroll
        for (int e = 0; e < NRH; ++e) {
          const float mu = m_run[e] == -INFINITY ? 0.f : m_run[e];
          s[e] = ex2(fmaf(s[e], c, -mu));
          l_part[e] += s[e];
        }
        // P^T row of this position (its NRH rows, 16 bytes per 8 rows): the
        // buffer is free once P . V of tile gj - PBUF is done
        const int pb = gj % Cfg::PBUF;
        if (gj >= Cfg::PBUF) {
          ok = warp_wait(&pv_done[pb], (uint32_t)((gj / Cfg::PBUF) - 1) & 1u, p.timeout_ns);
          if (!ok) break;
        }
        const uint32_t prow = smem_u32(sP + (size_t)pb * Cfg::P_BYTES) + (uint32_t)(kt * Cfg::P_ROW);
#pragma unroll
        for (int k = 0; k < NRH / 8; ++k) {
          const uint32_t a = prow + ((uint32_t)Cfg::p_chunk(kt, (row0 >> 3) + k) << 4);
          uint32_t w[4], wl[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            // (fp8: the block's V scale folded into the weights)
            const float a0 = s[8 * k + 2 * q] * vsc, a1 = s[8 * k + 2 * q + 1] * vsc;
            if constexpr (Cfg::BF) {
              w[q] = pack_bf16x2(a0, a1);
              wl[q] = pack_bf16x2(a0 - __uint_as_float(w[q] << 16), a1 - __uint_as_float(w[q] & 0xffff0000u));
            } else {
              w[q] = pack_f16x2(a0, a1);
            }
          }
          sts128(a, make_uint4(w[0], w[1], w[2], w[3]));
          if constexpr (Cfg::BF) sts128(a + Cfg::P_PART, make_uint4(wl[0], wl[1], wl[2], wl[3]));
        }
        fence_proxy_async();
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[pb]);
        if constexpr (Cfg::FP8) {
          // V of the next tile into the ring slot P . V(gj - 1) read
          if (gj + 1 < ntiles) {
            if (gj >= 1) {
              ok = warp_wait(&pv_done[(gj - 1) % Cfg::PBUF], (uint32_t)((gj - 1) / Cfg::PBUF) & 1u, p.timeout_ns);
              if (!ok) break;
            }
            if (!(ok = widen(gj + 1, true))) break;
          }
        }
      }
      if (!ok) break;
      if (staged) release_q((si + 1) % Cfg::QBUF, true);
      // ---- epilogue of the segment: O^T / l, or a normalised partial and its lse ----
      const int gl = g + n - 1;
      ok = warp_wait(&pv_done[gl % Cfg::PBUF], (uint32_t)(gl / Cfg::PBUF) & 1u, p.timeout_ns);
      if (ok) {  // row sums over the 128 positions (l_part is reset for the next segment)
        const float lrow = reduce_scatter<NRH, false>(l_part, lane);
        if (lane < NRH) red_l[hf][qd][lane] = lrow;
        __syncwarp();
        if (lane == 0) mbar_arrive(&xl[hf]);
        ok = warp_wait(&xl[hf], (uint32_t)si & 1u, p.timeout_ns);
      }
      if (!ok) break;
      tc::fence_after();
      const float lt = red_l[hf][0][rr] + red_l[hf][1][rr] + red_l[hf][2][rr] + red_l[hf][3][rr];
      uint32_t o[NRH];
      ld_cols<NRH>(tbase + lane_base + Cfg::COL_O + (uint32_t)(ob * Cfg::NPV + row0), o);
      // O^T is in registers: two segments on, P . V may overwrite the buffer
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&o_free[ob]);
      const int d = kt;  // O^T lane = head-dim index
      if (sg.whole) {
#pragma unroll
        for (int e = 0; e < NRH; ++e) {
          const int r = row0 + e;
          const float L = __shfl_sync(kFull, lt, e);
          if (r < p.R) {
            const int ii = r / p.G, gq = r - ii * p.G;
            const size_t idx = (((size_t)sg.b * p.q_len + ii) * p.Hq + sg.h * p.G + gq) * Cfg::D + d;
            const float v = L > 0.f ? __uint_as_float(o[e]) / L : 0.f;  // a row that sees nothing gives 0
            if constexpr (Cfg::OUT_BF)
              store_scalar(BF16{}, p.out, idx, v);
            else
              store_scalar(F16{}, p.out, idx, v);
          }
        }
      } else {
        const size_t part = (size_t)blockIdx.x * 2 + sg.slot;
        float *po = p.part_o + part * kMqRows * Cfg::D;
        float mine = -INFINITY;  // lse of row row0 + lane (lanes < NRH)
#pragma unroll
        for (int e = 0; e < NRH; ++e) {
          const float L = __shfl_sync(kFull, lt, e);
          po[(size_t)(row0 + e) * Cfg::D + d] = L > 0.f ? __uint_as_float(o[e]) / L : 0.f;
          if (lane == e && L > 0.f) mine = (m_run[e] == -INFINITY ? 0.f : m_run[e]) + log2f(L);
        }
        if (qd == 0 && lane < NRH) p.part_lse[part * kMqRows + row0 + lane] = mine;
      }
      g += n;
      ++si;
      sg = nx;
      have = nhave;
      nhave = have && wk.next(p, nx);
    }
    if (ok) {
      // sequences with no tile (no visible position for any new token): zeros,
      // sequence b by CTA b mod grid
      const size_t per_seq = (size_t)p.q_len * p.Hq * Cfg::D / 8;
      for (int b = blockIdx.x; b < B; b += gridDim.x)
        if (mq_seq(p, b).T == 0) {
          uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.out) + (size_t)b * per_seq * 8);
          for (size_t i = tid; i < per_seq; i += Cfg::SOFTMAX) dst[i] = make_uint4(0, 0, 0, 0);
        }
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
  } else if ((warp == Cfg::PRODUCER || warp == Cfg::V_PRODUCER) && lane == 0) {  // copies issued, never consumed
    if constexpr (Cfg::FP8) {  // the raw copies last issued into each slot (the f16 rings are written by this CTA)
      for (int j = kr_issued > Cfg::KRAW ? kr_issued - Cfg::KRAW : 0; j < kr_issued; ++j)
        mbar_wait_bounded(&kr_full[j % Cfg::KRAW], (uint32_t)(j / Cfg::KRAW) & 1u, p.timeout_ns);
      for (int j = vr_issued > Cfg::VRAW ? vr_issued - Cfg::VRAW : 0; j < vr_issued; ++j)
        mbar_wait_bounded(&vr_full[j % Cfg::VRAW], (uint32_t)(j / Cfg::VRAW) & 1u, p.timeout_ns);
    } else {
    for (int j = k_consumed; j < k_issued; ++j)
      mbar_wait_bounded(&k_full[j % Cfg::KSTAGES], (uint32_t)(j / Cfg::KSTAGES) & 1u, p.timeout_ns);
    for (int j = v_consumed; j < v_issued; ++j)
      mbar_wait_bounded(&v_full[j % Cfg::VSTAGES], (uint32_t)(j / Cfg::VSTAGES) & 1u, p.timeout_ns);
    }
  } else if (tid < Cfg::SOFTMAX) {
    asm volatile("cp.async.wait_all;" ::: "memory");  // a Q copy left in flight by an abort
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == Cfg::ISSUER) tc::dealloc(tbase, Cfg::TMEM_COLS);
  if (tid == 0) p.cta_flags[blockIdx.x] = cta_flags;
  grid_dep_launch();
}

// Finishes the items cut by range ends: block c takes the boundary between
// CTAs c and c + 1 and, if it falls inside an item and is that item's first,
// merges the partials of the item written by the CTAs c .. wl whose ranges
// are not empty (a CTA whose range starts at or after the item's first tile
// wrote slot 0, the one before slot 1) — weights 2^(lse - max lse), rows
// every partial leaves empty give 0.  Block 0 also publishes the call's
// status bits (the OR of every CTA's).
__global__ void __launch_bounds__(256) mq_merge_kernel(const MqParams p, int P, int out_bf16) {
  grid_dep_wait();
  if (blockIdx.x == 0 && threadIdx.x < 32) {
    int f = 0;
    for (int c = threadIdx.x; c < P; c += 32) f |= p.cta_flags[c];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) f |= __shfl_xor_sync(kFull, f, off);
    if (threadIdx.x == 0) *p.status = f;
  }
  const int c = blockIdx.x;
  const int W = p.prefix[p.B];
  if (c + 1 >= P || W <= 0) return;
  const int tcut = (int)((int64_t)W * (c + 1) / P);
  if (tcut <= 0 || tcut >= W) return;
  int lo = 0, hi = p.B;  // the sequence holding tile tcut
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.prefix[mid] <= tcut) lo = mid;
    else hi = mid - 1;
  }
  const int b = lo, base = p.prefix[b];
  const int T = (p.prefix[b + 1] - base) / p.Hkv;
  const int h = (tcut - base) / T;
  const int a = base + h * T, e = a + T;  // the item's tiles
  if (tcut == a) return;                          // the cut falls between items
  if ((int)((int64_t)W * c / P) > a) return;      // an earlier cut inside the item merges it
  const int wl = (int)(((int64_t)e * P - 1) / W);  // the CTA holding the item's last tile
  constexpr int D = kMqHeadDim;
  for (int i = threadIdx.x; i < p.R * (D / 4); i += blockDim.x) {
    const int r = i / (D / 4), d = 4 * (i % (D / 4));
    float M = -INFINITY;
    for (int w = c; w <= wl; ++w) {
      const int w0 = (int)((int64_t)W * w / P);
      if (w0 == (int)((int64_t)W * (w + 1) / P)) continue;  // an empty range (fewer tiles than CTAs)
      M = fmaxf(M, p.part_lse[((size_t)w * 2 + (w0 >= a ? 0 : 1)) * kMqRows + r]);
    }
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float den = 0.f;
    if (M != -INFINITY) {
      for (int w = c; w <= wl; ++w) {
        const int w0 = (int)((int64_t)W * w / P);
        if (w0 == (int)((int64_t)W * (w + 1) / P)) continue;
        const size_t part = (size_t)w * 2 + (w0 >= a ? 0 : 1);
        const float l = p.part_lse[part * kMqRows + r];
        if (l == -INFINITY) continue;
        const float wt = exp2f(l - M);
        const float4 o = *reinterpret_cast<const float4 *>(p.part_o + (part * kMqRows + r) * D + d);
        acc.x = fmaf(wt, o.x, acc.x);
        acc.y = fmaf(wt, o.y, acc.y);
        acc.z = fmaf(wt, o.z, acc.z);
        acc.w = fmaf(wt, o.w, acc.w);
        den += wt;
      }
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    const int ii = r / p.G, gq = r - ii * p.G;
    const size_t idx = (((size_t)b * p.q_len + ii) * p.Hq + h * p.G + gq) * D + d;
    const uint2 v = out_bf16 ? make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv))
                             : make_uint2(pack_f16x2(acc.x * inv, acc.y * inv), pack_f16x2(acc.z * inv, acc.w * inv));
    *reinterpret_cast<uint2 *>(static_cast<uint16_t *>(p.out) + idx) = v;
  }
}

static inline size_t mq_align(size_t x) { return (x + 255) / 256 * 256; }

MqWsLayout mq_ws_layout(int B, int grid) {
  MqWsLayout L;
  size_t o = mq_align(sizeof(WsHeader));
  L.prefix = o;
  o = mq_align(o + sizeof(int32_t) * (size_t)(B + 1));
  L.cta_flags = o;
  o = mq_align(o + sizeof(int32_t) * (size_t)grid);
  L.part_o = o;
  o = mq_align(o + sizeof(float) * (size_t)grid * 2 * kMqRows * kMqHeadDim);
  L.part_lse = o;
  o = mq_align(o + sizeof(float) * (size_t)grid * 2 * kMqRows);
  L.total = o;
  return L;
}

template <class Cfg>
static cudaError_t launch_mq_cfg(const MqParams &p, const CUtensorMap &tmK, const CUtensorMap &tmV, int grid,
                                 cudaStream_t stream) {
  static int configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorNotSupported;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(mq_decode_kernel<Cfg>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg::SMEM);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(Cfg::THREADS);
  cfg.dynamicSmemBytes = Cfg::SMEM;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, mq_decode_kernel<Cfg>, p, tmK, tmV);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t mc = {};
  mc.gridDim = dim3((unsigned)(grid > 1 ? grid - 1 : 1));
  mc.blockDim = dim3(256);
  mc.stream = stream;
  mc.attrs = attr;
  mc.numAttrs = 1;
  return cudaLaunchKernelEx(&mc, mq_merge_kernel, p, grid, Cfg::OUT_BF ? 1 : 0);
}

template <class T, class QT = T>
static cudaError_t launch_mq_rows(const MqParams &p, const CUtensorMap &tmK, const CUtensorMap &tmV, int grid,
                                  cudaStream_t stream) {
  if (p.R <= 16) return launch_mq_cfg<MqCfg<T, 8, QT>>(p, tmK, tmV, grid, stream);
  if (p.R <= 32) return launch_mq_cfg<MqCfg<T, 16, QT>>(p, tmK, tmV, grid, stream);
  if constexpr (T::kBytes == 1)
    return cudaErrorNotSupported;  // fp8: up to 32 rows
  else
    return launch_mq_cfg<MqCfg<T, 32, QT>>(p, tmK, tmV, grid, stream);
}

cudaError_t launch_mq_decode(const MqParams &p, int cache_dtype, int q_dtype, const CUtensorMap &tmK,
                             const CUtensorMap &tmV, int grid, cudaStream_t stream) {
  if (p.R < 1 || p.R > kMqRows || p.B < 1 || p.B > kMqMaxBatch || grid < 1) return cudaErrorNotSupported;
  if (cache_dtype == PKV_BF16) return launch_mq_rows<BF16>(p, tmK, tmV, grid, stream);
  if (cache_dtype == PKV_F16) return launch_mq_rows<F16>(p, tmK, tmV, grid, stream);
  if (cache_dtype == PKV_FP8_E4M3 && p.R <= kMqRowsFp8) {
    if (q_dtype == PKV_BF16) return launch_mq_rows<E4M3, BF16>(p, tmK, tmV, grid, stream);
    if (q_dtype == PKV_F16) return launch_mq_rows<E4M3, F16>(p, tmK, tmV, grid, stream);
  }
  return cudaErrorNotSupported;
}

}  // namespace pkv
