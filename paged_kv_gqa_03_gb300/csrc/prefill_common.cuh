// prefill_common.cuh — pieces shared by the two tcgen05 prefill kernels
// (prefill.cu: one persistent CTA per SM walking many work items;
// prefill_tiles.cu: one CTA per work item): the tile configuration, bounded
// warp-wide barrier waits and the softmax arithmetic helpers.
//
// The computation is FlashAttention's tiled form ("LLM推理优化实战" §3.2
// flash_attention: Q in row blocks, K / V in blocks of 128 positions, online
// softmax with running max m and sum l, O rescaled by exp(m_old - m_new)) with
// the causal mask of "苦猿的大模型日记 Day45" PART 04.  The tile pipeline both
// kernels run:
//  * K / V tiles of 128 positions = 8 paged blocks, fetched by TMA through the
//    block table (one 2 KiB box per block and 64-element panel) into a 2-deep
//    K ring and a 3-deep V ring: a K slot frees as soon as S = Q . K^T has
//    read it, a V slot when P . V has (V, read later, gets the deeper ring:
//    0.8 % faster than 3 + 2 on chunked prefill);
//  * S (128 x 128, f32) and O (128 x D, f32) live in tensor memory; S has three
//    buffers, and each buffer's P (the 16-bit weights) is written back over
//    the S columns its thread has read, so P . V takes A from tensor memory
//    (tcgen05.mma A-in-TMEM) and B = V from shared memory (128-byte swizzle,
//    MN-major); Q and K are 128-byte-swizzled K-major operands;
//  * eight softmax warps: thread (row, half) owns half of one query row's
//    columns (tcgen05.ld / st 32x32b; warps w and w + 4 share a lane
//    quarter); the halves exchange their partial row max once per tile;
//  * O is rescaled in tensor memory only when a row's running max grows by
//    more than 8 (log2 units): the result is exact either way, since P and l
//    share the stale max, and p <= 2^8 keeps P well inside 16-bit range;
//  * P . V takes P in the cache's 16-bit type (kind::f16 takes one type for
//    A and B, and V is read as the TMA lands it).  P needs more than bf16's 8
//    significant bits for the 2e-3 output bound, so for a bf16 cache P goes
//    in as a bf16 high part plus its bf16 residual (two MMAs per k-step, ~16
//    significant bits), written over the thread's S columns (high parts in
//    the first 32 of a half's 64 columns, residuals in the other 32); an f16
//    cache takes f16 P.  V is used exactly as stored, over bf16's whole range;
//    stale rows past a context are zeroed in shared memory before P . V;
//  * warp roles: 0-7 softmax + epilogue, 8 and 10 TMA producers of the K and
//    the V tiles (one warp issuing both tensors' copies spent much of each
//    tile period inside its issues), 9 S issue and tensor-memory allocation,
//    11 P . V issue (S waits only for K and for its buffer's last P . V,
//    P . V only for V and P: neither stream waits behind the other's inputs).  Every wait is bounded; a timeout sets
//    PKV_FLAG_TIMEOUT, the CTA drains its copies and MMAs and frees its tensor
//    memory;
//  * the softmax's per-column work runs two columns per instruction on the
//    packed f32x2 arithmetic of sm_100 and later, with a three-input max
//    (p_pair); the epilogue stages each warp's output rows in shared memory
//    so that its global stores cover whole half-rows (store_rows_staged).
#pragma once

#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace pkv {

template <class T, int D_>
struct PrefillCfg {
  static constexpr int D = D_;
  static constexpr bool BF = T::kCode == PKV_BF16;
  // P . V in the cache's type: for bf16, P as a high part plus its residual
  static constexpr int PARTS = BF ? 2 : 1;
  static constexpr int M = 128;                         // query rows per CTA
  static constexpr int N = 128;                         // cache positions per K / V tile
  static constexpr int BLOCKS = N / kBlock;             // paged blocks per tile
  static constexpr int PANELS = D / 64;                 // 128-byte panels per row
  static constexpr int PANEL_Q = M * 128;               // one Q panel (128 rows)
  static constexpr int PANEL_KV = N * 128;              // one K or V panel (128 positions)
  static constexpr int Q_BYTES = PANELS * PANEL_Q;
  static constexpr int KV_BYTES = PANELS * PANEL_KV;    // one K (or V) tile
  static constexpr int KSTAGES = 2, VSTAGES = 3;
  static constexpr int LOADS = BLOCKS * PANELS;         // TMA boxes per K (or V) tile
  static constexpr size_t SMEM = 1024 + Q_BYTES + (size_t)(KSTAGES + VSTAGES) * KV_BYTES;
  static constexpr int SBUF = 3;                        // S / P buffers in tensor memory
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_O = SBUF * N;           // O after the S buffers
  static constexpr int SOFTMAX = 256;                   // threads: 128 rows x 2 halves
  static constexpr int THREADS = SOFTMAX + 128;         // + K producer, S issue, V producer, P . V issue warps
  static constexpr int PRODUCER = SOFTMAX / 32, ISSUER = PRODUCER + 1, V_PRODUCER = PRODUCER + 2,
                       PV_ISSUER = PRODUCER + 3;  // warp ids
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(COL_O + D <= TMEM_COLS, "tensor memory");
  static_assert(LOADS <= 32, "one box per producer lane");
  static_assert(SMEM + 4096 <= 232448, "shared memory");
};

// A bounded wait whose outcome is the same for every lane of the warp (the
// tensor-memory loads and arrivals that follow are warp-collective).
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
  return __all_sync(kFull, mbar_wait_bounded(bar, parity, limit_ns));
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Two f32 values as one 64-bit register pair, for the packed f32x2
// arithmetic of sm_100 and later (one instruction issue for both lanes).
__device__ __forceinline__ uint64_t f2_pack(float x, float y) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(x), "f"(y));
  return r;
}
__device__ __forceinline__ float2 f2_unpack(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// max(a, b, c) in one instruction (sm_100 and later); like fmaxf, a NaN
// operand loses to a number.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// The softmax weights of two adjacent S columns, p = 2^(s * c - mu):
// `cmu` = {c, c} and `nmu` = {-mu, -mu} as f32x2 pairs, the two weights added
// lane-wise into `sum` (two partial row sums), and the pair packed as the
// cache's 16-bit type into `hi` — for bf16 with the residuals p - bf16(p),
// themselves rounded to bf16, in `lo` (~16 significant bits together).
template <bool BF>
__device__ __forceinline__ void p_pair(uint32_t s0, uint32_t s1, uint64_t cmu, uint64_t nmu, uint64_t &sum,
                                       uint32_t &hi, uint32_t &lo) {
  const float2 t = f2_unpack(f2_fma(f2_pack(__uint_as_float(s0), __uint_as_float(s1)), cmu, nmu));
  const float a0 = ex2(t.x), a1 = ex2(t.y);
  const uint64_t a = f2_pack(a0, a1);
  sum = f2_add(sum, a);
  if constexpr (BF) {
    const __nv_bfloat162 hp = __floats2bfloat162_rn(a0, a1);
    hi = *reinterpret_cast<const uint32_t *>(&hp);
    // the two rounded values back in f32: bf16 is the upper half of an f32
    const uint64_t h = f2_pack(__uint_as_float(hi << 16), __uint_as_float(hi & 0xffff0000u));
    const float2 r = f2_unpack(f2_sub(a, h));
    lo = pack_bf16x2(r.x, r.y);
  } else {
    hi = pack_f16x2(a0, a1);
    lo = 0u;
  }
}

template <bool BF>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (BF)
    return pack_bf16x2(lo, hi);
  else
    return pack_f16x2(lo, hi);
}

// S = Q . K^T of one K tile into tensor-memory columns dS: D / 16 MMAs over
// K-major, 128-byte-swizzled Q (at q0) and K (at k0) panels; issued by one
// thread.
template <class Cfg>
__device__ __forceinline__ void mma_s_tile(uint32_t dS, uint32_t q0, uint32_t k0) {
  constexpr uint32_t idS = tc::idesc_f16(Cfg::BF, Cfg::M, Cfg::N, false);
#pragma unroll
  for (int k = 0; k < Cfg::D / 16; ++k) {
    const uint32_t off = (uint32_t)((k >> 2) * Cfg::PANEL_Q + (k & 3) * 32);
    const uint32_t offk = (uint32_t)((k >> 2) * Cfg::PANEL_KV + (k & 3) * 32);
    tc::mma_f16(dS, tc::desc_sw128(q0 + off, 16, 1024), tc::desc_sw128(k0 + offk, 16, 1024), idS,
                k > 0 ? 1u : 0u);
  }
}

// O (+)= P . V of one V tile: P (f16 pairs) from the S buffer's tensor
// memory at pb, V (f16, MN-major, at v0) from shared memory.  `accumulate`
// false starts O afresh.  Issued by one thread.
template <class Cfg>
__device__ __forceinline__ void mma_pv_tile(uint32_t dO, uint32_t pb, uint32_t v0, bool accumulate) {
  constexpr uint32_t idO = tc::idesc_f16(Cfg::BF, Cfg::M, Cfg::D, true);  // P and V of the cache's type
#pragma unroll
  for (int k = 0; k < Cfg::N / 16; ++k) {
    // positions 16k .. 16k + 15: half k / 4 of the row, packed pairs (bf16:
    // the high parts, the residuals 32 columns further)
    const uint32_t pcol = (uint32_t)((k >> 2) * (Cfg::N / 2) + (k & 3) * 8);
    const uint64_t dv = tc::desc_sw128(v0 + (uint32_t)k * 2048, Cfg::PANEL_KV, 1024);
#pragma unroll
    for (int part = 0; part < Cfg::PARTS; ++part)
      tc::mma_f16_tmem_a(dO, pb + pcol + (uint32_t)(part * 32), dv, idO, (accumulate || k > 0 || part > 0) ? 1u : 0u);
  }
}

// Warp-wide: zeroes rows [z0, z1) of a V tile in shared memory (stale cache
// rows past a context inside its last block: their weights are 0, but 0 * NaN
// would still poison P . V), then makes the writes visible to the tensor core.
template <class Cfg>
__device__ __forceinline__ void zero_v_rows(uint8_t *vt, int z0, int z1, int lane) {
  if (z0 >= 0 && z0 < z1) {
    for (int idx = lane; idx < (z1 - z0) * 8 * Cfg::PANELS; idx += 32) {
      const int r = z0 + idx / (8 * Cfg::PANELS), rest = idx % (8 * Cfg::PANELS);
      sts128(smem_u32(vt + (rest >> 3) * Cfg::PANEL_KV + r * 128 + (rest & 7) * 16), make_uint4(0, 0, 0, 0));
    }
    fence_proxy_async();
  }
}

// Warp-wide: writes this thread's half output row — the D / 2 values `o` of
// O times `inv`, in the cache's 16-bit type — to `dst` (null: not stored)
// through 2 KiB of shared memory at `stage`.  Stored directly, each 16-byte
// store of a warp would touch 32 rows' lines; staged and read back
// transposed, each store covers whole half-rows (4 at D = 128, 8 at D = 64),
// one line per 128 bytes.  The warp's 32 half-rows of CH 16-byte chunks go
// through in passes of RP rows; 16-byte unit u of a pass sits at unit
// (u & ~7) | ((u ^ (u >> 3)) & 7), so 8 rows writing one chunk and a row's
// chunks read by 8 lanes hit distinct banks.
template <class Cfg>
__device__ __forceinline__ void store_rows_staged(const uint32_t (&o)[Cfg::D / 64][32], float inv, uint4 *dst,
                                                  uint8_t *stage, int lane) {
  constexpr int CH = Cfg::D / 16, RP = 2048 / (CH * 16), RPI = 32 / CH;
  auto unit = [](int u) { return (u & ~7) | ((u ^ (u >> 3)) & 7); };
#pragma unroll
  for (int pass = 0; pass < 32 / RP; ++pass) {
    if (lane / RP == pass) {
      const int lr = lane - pass * RP;
#pragma unroll
      for (int ch = 0; ch < CH; ++ch) {
        const uint32_t *src = &o[ch / 4][(ch % 4) * 8];
        uint32_t wv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          wv[e] = pack2<Cfg::BF>(__uint_as_float(src[2 * e]) * inv, __uint_as_float(src[2 * e + 1]) * inv);
        sts128(smem_u32(stage + unit(lr * CH + ch) * 16), make_uint4(wv[0], wv[1], wv[2], wv[3]));
      }
    }
    __syncwarp();
#pragma unroll
    for (int i = 0; i < RP / RPI; ++i) {
      const int lr = i * RPI + lane / CH, ch = lane % CH;
      uint4 *d =
          reinterpret_cast<uint4 *>(__shfl_sync(kFull, reinterpret_cast<unsigned long long>(dst), pass * RP + lr));
      const uint4 v = lds128(smem_u32(stage + unit(lr * CH + ch) * 16));
      if (d) d[ch] = v;
    }
    __syncwarp();
  }
}

// Warp-wide: multiplies this thread's OC columns of O (tensor memory at ta)
// by alpha.
template <class Cfg>
__device__ __forceinline__ void scale_o(uint32_t ta, float alpha) {
  constexpr int OC = Cfg::D / 2;
#pragma unroll
  for (int q = 0; q < OC / 32; ++q) {
    uint32_t o[32];
    tc::ld32(ta + (uint32_t)(q * 32), o);
#pragma unroll
    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
    tc::st32(ta + (uint32_t)(q * 32), o);
  }
}

}  // namespace pkv
