// common.cuh — device helpers shared by the sm_103a kernels of libpagedkv:
// inline PTX for mbarriers, TMA tensor loads, ldmatrix / movmatrix / mma.sync,
// the 128-byte shared-memory swizzle, and element conversions.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"
#include "pagedkv.h"

namespace pkv {

constexpr unsigned kFull = 0xffffffffu;

// ---------------------------------------------------------------------------
// Element types.  Tags carry the storage size; loads convert to fp32.
// ---------------------------------------------------------------------------
struct F32 { static constexpr int kBytes = 4; static constexpr int kCode = PKV_F32; };
struct F16 { static constexpr int kBytes = 2; static constexpr int kCode = PKV_F16; };
struct BF16 { static constexpr int kBytes = 2; static constexpr int kCode = PKV_BF16; };
struct E4M3 { static constexpr int kBytes = 1; static constexpr int kCode = PKV_FP8_E4M3; };

__device__ __forceinline__ float2 unpack2(F16, uint32_t w) {
  __half2 h = *reinterpret_cast<__half2 *>(&w);
  return __half22float2(h);
}
__device__ __forceinline__ float2 unpack2(BF16, uint32_t w) {
  __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162 *>(&w);
  return __bfloat1622float2(h);
}
// two e4m3 bytes (low 16 bits of w) -> two floats, via CUDA's fp8 conversion
__device__ __forceinline__ float2 unpack2_e4m3(uint16_t w) {
  __half2_raw r = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w), __NV_E4M3);
  __half2 h = *reinterpret_cast<__half2 *>(&r);
  return __half22float2(h);
}
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t w) {
  __half2_raw r = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w), __NV_E4M3);
  return *reinterpret_cast<uint32_t *>(&r);
}

__device__ __forceinline__ float load_scalar(F32, const void *p, size_t i) {
  return reinterpret_cast<const float *>(p)[i];
}
__device__ __forceinline__ float load_scalar(F16, const void *p, size_t i) {
  return __half2float(reinterpret_cast<const __half *>(p)[i]);
}
__device__ __forceinline__ float load_scalar(BF16, const void *p, size_t i) {
  return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p)[i]);
}

__device__ __forceinline__ void store_scalar(F32, void *p, size_t i, float v) {
  reinterpret_cast<float *>(p)[i] = v;
}
__device__ __forceinline__ void store_scalar(F16, void *p, size_t i, float v) {
  reinterpret_cast<__half *>(p)[i] = __float2half_rn(v);
}
__device__ __forceinline__ void store_scalar(BF16, void *p, size_t i, float v) {
  reinterpret_cast<__nv_bfloat16 *>(p)[i] = __float2bfloat16_rn(v);
}

__device__ __forceinline__ void store_out(int dtype, void *p, size_t i, float v) {
  if (dtype == PKV_F32) store_scalar(F32{}, p, i, v);
  else if (dtype == PKV_F16) store_scalar(F16{}, p, i, v);
  else store_scalar(BF16{}, p, i, v);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}

// ---------------------------------------------------------------------------
// Shared-memory addressing.  A (block, kv-head) tile is 16 token rows of
// ROWB = D * elem bytes.  TMA writes it with the 128-byte swizzle: each
// 128-byte line keeps its 16-byte chunks XOR-permuted by (line % 8).  Rows of
// >= 128 bytes are split into 128-byte-wide boxes of 16 lines (2 KiB each, box
// k at byte 2048*k); 64-byte rows pack two tokens per line.
// ---------------------------------------------------------------------------
template <int ROWB>
__device__ __forceinline__ uint32_t tile_off(int t, int byte) {
  if constexpr (ROWB >= 128) {
    const int box = byte >> 7, in = byte & 127;
    return box * 2048 + t * 128 + ((((in >> 4) ^ t) & 7) << 4) + (in & 15);
  } else {
    const int lin = t * ROWB + byte, line = lin >> 7, in = lin & 127;
    return line * 128 + ((((in >> 4) ^ line) & 7) << 4) + (in & 15);
  }
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------
// mbarrier + TMA (inline PTX).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Waits for `parity` of `bar`; gives up after `limit_ns` of wall time and
// returns false (the caller records a timeout and stops).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 0 && global_timer_ns() - t0 > limit_ns) return false;
  }
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *tm) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tm)) : "memory");
}
// 2-D tiled TMA load of box (x, y) into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *tm, int x, int y, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Programmatic dependent launch controls (no-ops without the launch attribute).
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" :::); }

// ---------------------------------------------------------------------------
// Warp-level tensor-core pieces (m16n8k16, fp32 accumulate).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
template <bool kBF16>
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  if constexpr (kBF16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds16(uint32_t addr) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

}  // namespace pkv
