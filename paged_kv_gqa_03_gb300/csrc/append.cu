// append.cu — step a3 (append the new token's K/V through the slot mapping)
// and step a2 (copy-on-write block copy).
//
// Append: k_cache[slot / 16][h][slot % 16][:] = k_new[b][h][:] — the cache
// update of incremental decoding ("大模型推理加速——KV Cache篇" §3.1 step 2;
// "苦猿的大模型日记 Day45" PART 02), addressed through the block table
// ("LLM推理优化实战" §2.2).  FP8 caches store e4m3(x / scale) with CUDA's
// saturating round-to-nearest-even conversion; a token at offset 0 opens its
// block and sets the block's scale to max|x| / 448 first.  When one call
// appends several tokens of a sequence (consecutive entries, positions in
// order), a later token of a block opened in the same call finds its opener at
// entry b - offset and derives the same scale from the opener's values, so it
// never reads the scale while the opener writes it.
#include "common.cuh"
#include "internal.h"

namespace pkv {

// One warp per (sequence, kv head, K-or-V).
template <class NewT, bool kFp8>
__global__ void __launch_bounds__(128)
    append_kernel(const void *__restrict__ k_new, const void *__restrict__ v_new, void *k_cache,
                  void *v_cache, float *k_scale, float *v_scale, const int64_t *__restrict__ slot_mapping,
                  int B, int Hkv, int D, int64_t num_blocks, int cache_esize) {
  grid_dep_wait();  // launched early behind the previous kernel; its writes are visible now
  const int gw = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (gw >= B * Hkv * 2) return;
  const int kv = gw & 1, bh = gw >> 1;
  const int b = bh / Hkv, h = bh % Hkv;
  const int64_t slot = slot_mapping[b];
  if (slot < 0) return;
  const int64_t blk = slot / kBlock;
  const int off = (int)(slot % kBlock);
  if (blk >= num_blocks) return;
  const void *src = kv ? v_new : k_new;
  void *cache = kv ? v_cache : k_cache;
  const size_t src_elem = ((size_t)b * Hkv + h) * D;
  const size_t dst_elem = ((size_t)(blk * Hkv + h) * kBlock + off) * D;
  if constexpr (!kFp8) {
    // bit-exact copy of D * esize bytes, 16 bytes per lane-step
    const uint4 *s16 = reinterpret_cast<const uint4 *>(static_cast<const uint8_t *>(src) + src_elem * cache_esize);
    uint4 *d16 = reinterpret_cast<uint4 *>(static_cast<uint8_t *>(cache) + dst_elem * cache_esize);
    for (int i = lane; i < D * cache_esize / 16; i += 32) d16[i] = s16[i];
  } else {
    float *scales = kv ? v_scale : k_scale;
    const size_t sidx = (size_t)blk * Hkv + h;
    const int epl = D / 32;  // 2 or 4 elements per lane
    float x[4];
    float amax = 0.f;
    for (int e = 0; e < epl; ++e) {
      x[e] = load_scalar(NewT{}, src, src_elem + lane * epl + e);
      amax = fmaxf(amax, fabsf(x[e]));
    }
    float scale;
    if (off == 0) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
      scale = amax > 0.f ? amax / 448.0f : 1.0f;
      if (lane == 0) scales[sidx] = scale;
    } else if (b >= off && slot_mapping[b - off] == blk * kBlock) {
      // the block's opener is entry b - off of this call: same scale, from its values
      const size_t osrc = ((size_t)(b - off) * Hkv + h) * D;
      float oa = 0.f;
      for (int e = 0; e < epl; ++e) oa = fmaxf(oa, fabsf(load_scalar(NewT{}, src, osrc + lane * epl + e)));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) oa = fmaxf(oa, __shfl_xor_sync(kFull, oa, o));
      scale = oa > 0.f ? oa / 448.0f : 1.0f;
    } else {
      scale = scales[sidx];
    }
    uint32_t packed = 0;
    for (int e = 0; e < epl; ++e) {
      const __nv_fp8_storage_t q = __nv_cvt_float_to_fp8(x[e] / scale, __NV_SATFINITE, __NV_E4M3);
      packed |= (uint32_t)q << (8 * e);
    }
    uint8_t *dst = static_cast<uint8_t *>(cache) + dst_elem + lane * epl;
    if (epl == 4)
      *reinterpret_cast<uint32_t *>(dst) = packed;
    else
      *reinterpret_cast<uint16_t *>(dst) = (uint16_t)packed;
  }
}

cudaError_t launch_append(const void *k_new, const void *v_new, int new_dtype, void *k_cache, void *v_cache,
                          int cache_dtype, float *k_scale, float *v_scale, const int64_t *slot_mapping, int B,
                          int Hkv, int D, int64_t num_blocks, cudaStream_t stream) {
  const int warps = B * Hkv * 2;
  if (warps == 0) return cudaSuccess;
  const int esize = cache_dtype == PKV_F32 ? 4 : (cache_dtype == PKV_FP8_E4M3 ? 1 : 2);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((warps + 3) / 4);
  cfg.blockDim = dim3(128);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = stream != nullptr ? 1 : 0;  // early launch on explicit streams only
  if (cache_dtype != PKV_FP8_E4M3)
    return cudaLaunchKernelEx(&cfg, append_kernel<F32, false>, k_new, v_new, k_cache, v_cache, k_scale, v_scale,
                              slot_mapping, B, Hkv, D, num_blocks, esize);
  if (new_dtype == PKV_F32)
    return cudaLaunchKernelEx(&cfg, append_kernel<F32, true>, k_new, v_new, k_cache, v_cache, k_scale, v_scale,
                              slot_mapping, B, Hkv, D, num_blocks, esize);
  if (new_dtype == PKV_F16)
    return cudaLaunchKernelEx(&cfg, append_kernel<F16, true>, k_new, v_new, k_cache, v_cache, k_scale, v_scale,
                              slot_mapping, B, Hkv, D, num_blocks, esize);
  return cudaLaunchKernelEx(&cfg, append_kernel<BF16, true>, k_new, v_new, k_cache, v_cache, k_scale, v_scale,
                            slot_mapping, B, Hkv, D, num_blocks, esize);
}

// ---------------------------------------------------------------------------
// Calibrated FP8 append: a block's scale is the smallest power of two p with
// max|x| <= 448 p over the block's tokens; a token that outgrows it raises it
// and re-quantises the block's earlier bytes, e4m3(fp32(decode(q) * p_old) /
// p_new) — an exact exponent shift in the e4m3 normal range — so no stored
// value saturates (the FP8 calibration that "苦猿的大模型日记 Day45" PART 02
// and "大模型推理加速核心KV Cache 复用机制与内存布局优化" §四 say decides quality).
// One warp per (run of consecutive entries in one block, kv head, K or V):
// the tokens of a run are applied in order, each lane owning the same head-dim
// bytes of every row, so earlier rows it re-quantises are its own writes.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float pow2_scale(float amax) {
  if (!(amax > 0.f)) return 1.f;
  int e;
  const float m = frexpf(amax, &e);  // amax = m * 2^e, 0.5 <= m < 1
  return ldexpf(1.f, m <= 0.875f ? e - 9 : e - 8);  // amax <= 448 * 2^k = 0.875 * 2^(9 + k)
}

template <class NewT>
__global__ void __launch_bounds__(128)
    append_calibrated_kernel(const void *__restrict__ k_new, const void *__restrict__ v_new, uint8_t *k_cache,
                             uint8_t *v_cache, float *k_scale, float *v_scale,
                             const int64_t *__restrict__ slot_mapping, int B, int Hkv, int D, int64_t num_blocks) {
  grid_dep_wait();
  const int gw = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (gw >= B * Hkv * 2) return;
  const int kv = gw & 1, bh = gw >> 1;
  const int b0 = bh / Hkv, h = bh % Hkv;
  const int64_t slot0 = slot_mapping[b0];
  if (slot0 < 0) return;
  const int64_t blk = slot0 / kBlock;
  if (blk >= num_blocks) return;
  // an entry that continues a run (the previous entry holds the previous
  // position of the same block) is applied by the run's first warp
  if (slot0 % kBlock != 0 && b0 > 0 && slot_mapping[b0 - 1] == slot0 - 1) return;
  const void *src = kv ? v_new : k_new;
  uint8_t *cache = kv ? v_cache : k_cache;
  float *scales = kv ? v_scale : k_scale;
  const size_t sidx = (size_t)blk * Hkv + h;
  uint8_t *tile = cache + (size_t)(blk * Hkv + h) * kBlock * D;
  const int epl = D / 32;  // bytes of a row owned by a lane (2 or 4)
  float sc = scales[sidx];
  for (int b = b0;; ++b) {
    const int off = (int)(slot_mapping[b] % kBlock);
    float x[4];
    float amax = 0.f;
    for (int e = 0; e < epl; ++e) {
      x[e] = load_scalar(NewT{}, src, ((size_t)b * Hkv + h) * D + lane * epl + e);
      amax = fmaxf(amax, fabsf(x[e]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
    const float cand = pow2_scale(amax);
    if (off == 0) {
      sc = cand;
    } else if (cand > sc) {
      for (int t = 0; t < off; ++t) {  // re-quantise this lane's bytes of rows 0 .. off-1
        uint8_t *row = tile + (size_t)t * D + lane * epl;
        for (int e = 0; e < epl; e += 2) {
          const uint16_t w = *reinterpret_cast<const uint16_t *>(row + e);
          const float2 v = unpack2_e4m3(w);
          const float r0 = __fdiv_rn(__fmul_rn(v.x, sc), cand), r1 = __fdiv_rn(__fmul_rn(v.y, sc), cand);
          const uint16_t q0 = __nv_cvt_float_to_fp8(r0, __NV_SATFINITE, __NV_E4M3);
          const uint16_t q1 = __nv_cvt_float_to_fp8(r1, __NV_SATFINITE, __NV_E4M3);
          *reinterpret_cast<uint16_t *>(row + e) = (uint16_t)(q0 | (q1 << 8));
        }
      }
      sc = cand;
    }
    uint8_t *dst = tile + (size_t)off * D + lane * epl;
    for (int e = 0; e < epl; ++e) dst[e] = (uint8_t)__nv_cvt_float_to_fp8(__fdiv_rn(x[e], sc), __NV_SATFINITE, __NV_E4M3);
    if (!(b + 1 < B && off + 1 < kBlock && slot_mapping[b + 1] == slot_mapping[b] + 1)) break;
  }
  if (lane == 0) scales[sidx] = sc;
}

cudaError_t launch_append_calibrated(const void *k_new, const void *v_new, int new_dtype, void *k_cache,
                                     void *v_cache, float *k_scale, float *v_scale, const int64_t *slot_mapping,
                                     int B, int Hkv, int D, int64_t num_blocks, cudaStream_t stream) {
  const int warps = B * Hkv * 2;
  if (warps == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((warps + 3) / 4);
  cfg.blockDim = dim3(128);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = stream != nullptr ? 1 : 0;
  uint8_t *kc = static_cast<uint8_t *>(k_cache), *vc = static_cast<uint8_t *>(v_cache);
  if (new_dtype == PKV_F32)
    return cudaLaunchKernelEx(&cfg, append_calibrated_kernel<F32>, k_new, v_new, kc, vc, k_scale, v_scale,
                              slot_mapping, B, Hkv, D, num_blocks);
  if (new_dtype == PKV_F16)
    return cudaLaunchKernelEx(&cfg, append_calibrated_kernel<F16>, k_new, v_new, kc, vc, k_scale, v_scale,
                              slot_mapping, B, Hkv, D, num_blocks);
  return cudaLaunchKernelEx(&cfg, append_calibrated_kernel<BF16>, k_new, v_new, kc, vc, k_scale, v_scale,
                            slot_mapping, B, Hkv, D, num_blocks);
}

// Copy-on-write: cache[dst] = cache[src] for all kv heads (one CTA per pair
// and K/V side), plus the block's fp8 scales.
__global__ void __launch_bounds__(256)
    copy_blocks_kernel(uint8_t *k_cache, uint8_t *v_cache, float *k_scale, float *v_scale,
                       const int32_t *__restrict__ pairs, int Hkv, size_t block_bytes, int64_t num_blocks) {
  const int pair = blockIdx.x, kv = blockIdx.y;
  const int src = pairs[2 * pair], dst = pairs[2 * pair + 1];
  if (src < 0 || dst < 0 || src >= num_blocks || dst >= num_blocks || src == dst) return;
  uint8_t *base = kv ? v_cache : k_cache;
  const uint4 *s = reinterpret_cast<const uint4 *>(base + (size_t)src * block_bytes);
  uint4 *d = reinterpret_cast<uint4 *>(base + (size_t)dst * block_bytes);
  for (size_t i = threadIdx.x; i < block_bytes / 16; i += blockDim.x) d[i] = s[i];
  float *sc = kv ? v_scale : k_scale;
  if (sc != nullptr)
    for (int h = threadIdx.x; h < Hkv; h += blockDim.x) sc[(size_t)dst * Hkv + h] = sc[(size_t)src * Hkv + h];
}

cudaError_t launch_copy_blocks(void *k_cache, void *v_cache, int cache_dtype, float *k_scale, float *v_scale,
                               const int32_t *pairs, int n_pairs, int Hkv, int D, int64_t num_blocks,
                               cudaStream_t stream) {
  if (n_pairs == 0) return cudaSuccess;
  const int esize = cache_dtype == PKV_F32 ? 4 : (cache_dtype == PKV_FP8_E4M3 ? 1 : 2);
  const size_t block_bytes = (size_t)Hkv * kBlock * D * esize;
  const bool fp8 = cache_dtype == PKV_FP8_E4M3;
  copy_blocks_kernel<<<dim3(n_pairs, 2), 256, 0, stream>>>(
      static_cast<uint8_t *>(k_cache), static_cast<uint8_t *>(v_cache), fp8 ? k_scale : nullptr,
      fp8 ? v_scale : nullptr, pairs, Hkv, block_bytes, num_blocks);
  return cudaGetLastError();
}

}  // namespace pkv
