// prefill.cu — paged prefill attention on the fifth-generation tensor cores
// (tcgen05): every new token of a sequence attends causally to the sequence's
// paged cache (its prompt and any cached prefix), optionally inside a sliding
// window.
//
// The computation is FlashAttention's tiled form ("LLM推理优化实战" §3.2
// flash_attention: Q in row blocks, K / V in blocks of 128 positions, online
// softmax with running max m and sum l, O rescaled by exp(m_old - m_new)) with
// the causal mask of "苦猿的大模型日记 Day45" PART 04.  GB300 design:
//  * one CTA per (sequence, kv head, tile of 128 query rows); a row is (new
//    token i, query head g) of the kv head's group, token-major, so GQA heads
//    share every K / V tile;
//  * K / V tiles of 128 positions = 8 paged blocks, fetched by TMA through the
//    block table (one 2 KiB box per block and 64-element panel) into a
//    STAGES-deep ring;
//  * S = Q . K^T (128 x 128, f32) and O += P . V (128 x D, f32) are tcgen05.mma
//    with operands in shared memory (128-byte swizzle; V as an MN-major
//    operand) and accumulators in tensor memory; S is double-buffered so the
//    MMA of tile j+1 overlaps the softmax of tile j;
//  * four softmax warps own one query row per thread (tcgen05.ld 32x32b): the
//    row max needs no shuffles; P goes back to shared memory as the A operand;
//  * O is rescaled in tensor memory only when a row's running max grows by
//    more than 8 (log2 units): the result is exact either way, since P and l
//    share the stale max, and p <= 2^8 keeps P well inside 16-bit range;
//  * P must have V's type (kind::f16 takes one type for A and B).  f16 keeps
//    11 significant bits, enough for the 2e-3 output bound; bf16 keeps 8, so a
//    bf16 P goes in as a high part plus its bf16 residual, two MMAs on the
//    same V tile (the weights then carry ~16 bits);
//  * warp roles: 0-3 softmax + epilogue, 4 TMA producer, 5 MMA issue and
//    tensor-memory allocation.  Every wait is bounded; a timeout sets
//    PKV_FLAG_TIMEOUT, the CTA drains its copies and MMAs and frees its tensor
//    memory.
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace pkv {

template <class T, int D_>
struct PrefillCfg {
  static constexpr int D = D_;
  static constexpr bool BF = T::kCode == PKV_BF16;
  static constexpr int M = 128;                         // query rows per CTA
  static constexpr int N = 128;                         // cache positions per K / V tile
  static constexpr int BLOCKS = N / kBlock;             // paged blocks per tile
  static constexpr int PANELS = D / 64;                 // 128-byte panels per row
  static constexpr int PANEL_Q = M * 128;               // one Q or P panel (128 rows)
  static constexpr int PANEL_KV = N * 128;              // one K or V panel (128 positions)
  static constexpr int Q_BYTES = PANELS * PANEL_Q;
  static constexpr int KV_BYTES = PANELS * PANEL_KV;    // the K (or V) half of a stage
  static constexpr int STAGES = D == 64 ? 3 : 2;
  static constexpr int STAGE_BYTES = 2 * KV_BYTES;
  static constexpr bool SPLIT = BF;                      // P as bf16 high + residual
  static constexpr int P_PART = 2 * PANEL_Q;            // 128 rows x 128 positions
  static constexpr int P_BYTES = (SPLIT ? 2 : 1) * P_PART;
  static constexpr size_t SMEM = 1024 + Q_BYTES + (size_t)STAGES * STAGE_BYTES + P_BYTES;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_S = 0;                  // S buffers at columns 0 and 128
  static constexpr uint32_t COL_O = 256;                // O at columns 256 .. 256 + D
  static constexpr int THREADS = 192;
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(SMEM <= 232448, "shared memory");
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
template <bool BF>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (BF)
    return pack_bf16x2(lo, hi);
  else
    return pack_f16x2(lo, hi);
}

template <class Cfg>
__global__ void __launch_bounds__(Cfg::THREADS, 1)
    prefill_kernel(const __grid_constant__ PrefillParams p, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t *sQ = smem;
  uint8_t *sKV = sQ + Cfg::Q_BYTES;
  uint8_t *sP = sKV + (size_t)Cfg::STAGES * Cfg::STAGE_BYTES;
  __shared__ __align__(8) uint64_t full[Cfg::STAGES], empty[Cfg::STAGES];
  __shared__ __align__(8) uint64_t s_full[2], s_free[2], p_full, pv_done, fin;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag, cta_flags, consumed, issued;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile = p.max_tiles - 1 - (int)blockIdx.x;  // heaviest (latest) row tiles first
  const int h = blockIdx.y, b = blockIdx.z;
  const int qs = __ldg(p.q_start + b);
  const int n = __ldg(p.q_start + b + 1) - qs;
  if (tid == 0 && tile == 0 && (n > p.max_q_len || n < 0) && p.status) atomicOr(p.status, PKV_FLAG_BAD_LEN);
  const int R = n * p.G;  // query rows of this kv head
  const int r0 = tile * Cfg::M;
  if (n <= 0 || r0 >= R) return;  // the whole CTA: no barrier or tensor memory touched yet

  const int ctx_raw = __ldg(p.context_lens + b);
  const int ctx = ctx_raw < 0 ? 0 : (ctx_raw > p.max_blocks * kBlock ? p.max_blocks * kBlock : ctx_raw);
  const int nblk = (ctx + kBlock - 1) / kBlock;
  const int i_lo = r0 / p.G, i_hi = min(R - 1, r0 + Cfg::M - 1) / p.G;
  const int lim_lo = ctx - n + i_lo + 1, lim_hi = ctx - n + i_hi + 1;  // exclusive causal ends
  const int first = p.window > 0 ? max(0, lim_lo - p.window) : 0;
  const int j_first = first / Cfg::N;
  const int T = lim_hi > 0 ? (lim_hi - 1) / Cfg::N - j_first + 1 : 0;  // K / V tiles to stream

  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < Cfg::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    mbar_init(&s_free[0], 4);
    mbar_init(&s_free[1], 4);
    mbar_init(&p_full, 4);
    mbar_init(&pv_done, 1);
    mbar_init(&fin, 1);
    fence_barrier_init();
    abort_flag = 0;
    cta_flags = ctx_raw != ctx ? PKV_FLAG_BAD_LEN : 0;
    consumed = 0;
    issued = 0;
  }
  if (warp == 5) tc::alloc(&tmem_base, Cfg::TMEM_COLS);
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (tid < Cfg::M) {  // Q tile: each softmax thread stages its own row (zeros past R)
    const int r = r0 + tid;
    const int ii = r / p.G, g = r - ii * p.G;
    const uint4 *src = r < R ? reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(p.q) +
                                                             ((size_t)(qs + ii) * p.Hq + h * p.G + g) * Cfg::D)
                             : nullptr;
#pragma unroll
    for (int c = 0; c < Cfg::D / 8; ++c) {
      const uint4 v = src ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
      sts128(smem_u32(sQ + (c >> 3) * Cfg::PANEL_Q + tid * 128 + (((c & 7) ^ (tid & 7)) << 4)), v);
    }
    fence_proxy_async();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tbase = tmem_base;

  if (warp == 4) {
    // ---------------- TMA producer ----------------
    for (int j = 0; j < T; ++j) {
      const int st = j % Cfg::STAGES;
      if (j >= Cfg::STAGES &&
          !warp_wait(&empty[st], (uint32_t)((j / Cfg::STAGES) - 1) & 1u, p.timeout_ns)) {
        if (lane == 0) {
          atomicOr(&cta_flags, PKV_FLAG_TIMEOUT);
          abort_flag = 1;
        }
        break;
      }
      if (__any_sync(kFull, *(volatile int *)&abort_flag)) break;
      const int lb = (j_first + j) * Cfg::BLOCKS + (lane & (Cfg::BLOCKS - 1));
      int64_t trow = p.num_blocks * p.Hkv;  // past the tensor: TMA fills zeros
      if (lb < nblk) {
        const int id = __ldg(p.block_table + (size_t)b * p.max_blocks + lb);
        if (id >= 0 && (int64_t)id < p.num_blocks)
          trow = (int64_t)id * p.Hkv + h;
        else
          atomicOr(&cta_flags, PKV_FLAG_BAD_BLOCK);
      }
      if (lane == 0) mbar_arrive_expect_tx(&full[st], Cfg::STAGE_BYTES);
      __syncwarp();
      if (lane < 2 * Cfg::BLOCKS * Cfg::PANELS) {  // one box per lane: (block, K or V, panel)
        const int blk = lane & (Cfg::BLOCKS - 1), kv = (lane / Cfg::BLOCKS) & 1, panel = lane / (2 * Cfg::BLOCKS);
        uint8_t *dst = sKV + (size_t)st * Cfg::STAGE_BYTES + kv * Cfg::KV_BYTES + panel * Cfg::PANEL_KV + blk * 2048;
        tma_load_2d(dst, kv ? &tmV : &tmK, panel * 64, (int)(trow * kBlock), &full[st]);
      }
      if (lane == 0) issued = j + 1;
    }
  } else if (warp == 5) {
    // ---------------- MMA issue ----------------
    constexpr uint32_t idS = tc::idesc_f16(Cfg::BF, Cfg::M, Cfg::N, false);
    constexpr uint32_t idO = tc::idesc_f16(Cfg::BF, Cfg::M, Cfg::D, true);
    const uint32_t q0 = smem_u32(sQ), p0 = smem_u32(sP);
    bool ok = true;
    for (int j = 0; j <= T && ok; ++j) {
      if (j < T) {
        const int st = j % Cfg::STAGES;
        ok = warp_wait(&full[st], (uint32_t)(j / Cfg::STAGES) & 1u, p.timeout_ns);
        if (ok && j >= 2) ok = warp_wait(&s_free[j & 1], (uint32_t)((j >> 1) - 1) & 1u, p.timeout_ns);
        if (!ok) break;
        if (lane == 0) consumed = j + 1;
        uint8_t *kt = sKV + (size_t)st * Cfg::STAGE_BYTES;
        // stale cache rows past ctx inside the sequence's last block: zero them in V
        // (their weights are 0, but 0 * NaN would still poison P . V)
        const int kv0 = (j_first + j) * Cfg::N;
        const int z0 = ctx - kv0, z1 = min(nblk * kBlock - kv0, Cfg::N);
        if (z0 >= 0 && z0 < z1) {
          for (int idx = lane; idx < (z1 - z0) * 8 * Cfg::PANELS; idx += 32) {
            const int row = z0 + idx / (8 * Cfg::PANELS), rest = idx % (8 * Cfg::PANELS);
            sts128(smem_u32(kt + Cfg::KV_BYTES + (rest >> 3) * Cfg::PANEL_KV + row * 128 + (rest & 7) * 16),
                   make_uint4(0, 0, 0, 0));
          }
          fence_proxy_async();
        }
        __syncwarp();
        tc::fence_after();
        if (lane == 0) {
          const uint32_t k0 = smem_u32(kt);
          const uint32_t dS = tbase + Cfg::COL_S + (uint32_t)(j & 1) * Cfg::N;
#pragma unroll
          for (int k = 0; k < Cfg::D / 16; ++k) {
            const uint32_t off = (uint32_t)((k >> 2) * Cfg::PANEL_Q + (k & 3) * 32);
            const uint32_t offk = (uint32_t)((k >> 2) * Cfg::PANEL_KV + (k & 3) * 32);
            tc::mma_f16(dS, tc::desc_sw128(q0 + off, 16, 1024), tc::desc_sw128(k0 + offk, 16, 1024), idS,
                        k > 0 ? 1u : 0u);
          }
          tc::commit(&s_full[j & 1]);
        }
        __syncwarp();
      }
      if (j >= 1) {
        const int jp = j - 1, stp = jp % Cfg::STAGES;
        ok = warp_wait(&p_full, (uint32_t)jp & 1u, p.timeout_ns);
        if (!ok) break;
        tc::fence_after();
        if (lane == 0) {
          const uint32_t v0 = smem_u32(sKV + (size_t)stp * Cfg::STAGE_BYTES + Cfg::KV_BYTES);
#pragma unroll
          for (int k = 0; k < Cfg::N / 16; ++k) {
            const uint32_t offp = (uint32_t)((k >> 2) * Cfg::PANEL_Q + (k & 3) * 32);
            const uint64_t dv = tc::desc_sw128(v0 + (uint32_t)k * 2048, Cfg::PANEL_KV, 1024);
            tc::mma_f16(tbase + Cfg::COL_O, tc::desc_sw128(p0 + offp, 16, 1024), dv, idO,
                        (jp > 0 || k > 0) ? 1u : 0u);
            if constexpr (Cfg::SPLIT)
              tc::mma_f16(tbase + Cfg::COL_O, tc::desc_sw128(p0 + Cfg::P_PART + offp, 16, 1024), dv, idO, 1u);
          }
          tc::commit(&pv_done);
          tc::commit(&empty[stp]);
        }
        __syncwarp();
      }
      if (__any_sync(kFull, *(volatile int *)&abort_flag)) break;
    }
    if (!ok && lane == 0) {
      atomicOr(&cta_flags, PKV_FLAG_TIMEOUT);
      abort_flag = 1;
    }
  } else {
    // ---------------- softmax + epilogue (one query row per thread) ----------------
    const int r = r0 + tid;
    const bool valid = r < R;
    const int lim = valid ? ctx - n + r / p.G + 1 : 0;  // visible positions [lo, lim)
    const int lo = (valid && p.window > 0) ? max(0, lim - p.window) : 0;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const float c = p.scale_log2;
    float m_run = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < T; ++j) {
      ok = warp_wait(&s_full[j & 1], (uint32_t)(j >> 1) & 1u, p.timeout_ns);
      if (!ok) break;
      tc::fence_after();
      uint32_t s[Cfg::N / 32][32];
#pragma unroll
      for (int q = 0; q < Cfg::N / 32; ++q)
        tc::ld32(tbase + lane_base + Cfg::COL_S + (uint32_t)(j & 1) * Cfg::N + (uint32_t)q * 32, s[q]);
      tc::wait_ld();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[j & 1]);
      const int kv0 = (j_first + j) * Cfg::N;
      if (!(kv0 >= lo && kv0 + Cfg::N <= lim)) {  // a mask edge crosses this tile
#pragma unroll
        for (int q = 0; q < Cfg::N / 32; ++q)
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int pos = kv0 + q * 32 + e;
            if (pos < lo || pos >= lim) s[q][e] = 0xff800000u;  // -inf
          }
      }
      float mx = -INFINITY;
#pragma unroll
      for (int q = 0; q < Cfg::N / 32; ++q)
#pragma unroll
        for (int e = 0; e < 32; ++e) mx = fmaxf(mx, __uint_as_float(s[q][e]));
      const float m_new = fmaxf(m_run, mx * c);
      const bool need = m_new > m_run + 8.f;
      if (j > 0) {  // P . V of the previous tile has finished reading P and writing O
        ok = warp_wait(&pv_done, (uint32_t)(j - 1) & 1u, p.timeout_ns);
        if (!ok) break;
        tc::fence_after();
      }
      if (__any_sync(kFull, need)) {
        const float alpha = m_new == -INFINITY ? 1.f : ex2(m_run - m_new);
        if (j > 0) {
#pragma unroll
          for (int q = 0; q < Cfg::D / 32; ++q) {
            uint32_t o[32];
            tc::ld32(tbase + lane_base + Cfg::COL_O + (uint32_t)q * 32, o);
            tc::wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tc::st32(tbase + lane_base + Cfg::COL_O + (uint32_t)q * 32, o);
          }
          tc::wait_st();
        }
        l *= alpha;
        m_run = m_new;
      }
      const float mu = m_run == -INFINITY ? 0.f : m_run;
      float sum = 0.f;
#pragma unroll
      for (int ch = 0; ch < Cfg::N / 8; ++ch) {  // 16-byte chunks of the P row
        uint32_t w[4], wl[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int col = ch * 8 + 2 * e;
          const float a0 = ex2(fmaf(__uint_as_float(s[col >> 5][col & 31]), c, -mu));
          const float a1 = ex2(fmaf(__uint_as_float(s[(col + 1) >> 5][(col + 1) & 31]), c, -mu));
          sum += a0 + a1;
          w[e] = pack2<Cfg::BF>(a0, a1);
          if constexpr (Cfg::SPLIT) {
            const float2 hi = unpack2(BF16{}, w[e]);
            wl[e] = pack_bf16x2(a0 - hi.x, a1 - hi.y);
          }
        }
        const uint32_t off = (uint32_t)((ch >> 3) * Cfg::PANEL_Q + tid * 128 + (((ch & 7) ^ (tid & 7)) << 4));
        sts128(smem_u32(sP + off), make_uint4(w[0], w[1], w[2], w[3]));
        if constexpr (Cfg::SPLIT) sts128(smem_u32(sP + Cfg::P_PART + off), make_uint4(wl[0], wl[1], wl[2], wl[3]));
      }
      l += sum;
      fence_proxy_async();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full);
    }
    if (ok && T > 0) ok = warp_wait(&pv_done, (uint32_t)(T - 1) & 1u, p.timeout_ns);
    if (!ok) {
      if (lane == 0) {
        atomicOr(&cta_flags, PKV_FLAG_TIMEOUT);
        abort_flag = 1;
      }
    } else {
      tc::fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;  // a row that sees nothing gives 0
      const int ii = r / p.G, g = r - ii * p.G;
      uint4 *dst = valid ? reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.out) +
                                                     ((size_t)(qs + ii) * p.Hq + h * p.G + g) * Cfg::D)
                         : nullptr;
#pragma unroll
      for (int q = 0; q < Cfg::D / 32; ++q) {
        uint32_t o[32];
        if (T > 0) {
          tc::ld32(tbase + lane_base + Cfg::COL_O + (uint32_t)q * 32, o);
          tc::wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = 0u;
        }
        if (dst) {
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = pack2<Cfg::BF>(__uint_as_float(o[v * 8 + 2 * e]) * inv, __uint_as_float(o[v * 8 + 2 * e + 1]) * inv);
            dst[q * 4 + v] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
    }
  }

  // ---------------- drain, then free tensor memory ----------------
  tc::fence_before();
  __syncthreads();
  if (warp == 5) {
    if (lane == 0) tc::commit(&fin);  // completes once every issued MMA has
    __syncwarp();
    if (!mbar_wait_bounded(&fin, 0, p.timeout_ns) && lane == 0) atomicOr(&cta_flags, PKV_FLAG_TIMEOUT);
  } else if (warp == 4 && lane == 0) {
    for (int j = consumed; j < issued; ++j)  // copies issued but never consumed (abort only)
      mbar_wait_bounded(&full[j % Cfg::STAGES], (uint32_t)(j / Cfg::STAGES) & 1u, p.timeout_ns);
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == 5) tc::dealloc(tbase, Cfg::TMEM_COLS);
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
    e = cudaFuncSetAttribute(prefill_kernel<Cfg>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg::SMEM);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  const dim3 grid((unsigned)p.max_tiles, (unsigned)p.Hkv, (unsigned)p.B);
  prefill_kernel<Cfg><<<grid, Cfg::THREADS, Cfg::SMEM, stream>>>(p, tmK, tmV);
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
