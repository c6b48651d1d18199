// decode_static.cu — paged_decode_attention_static, the decode entry point for
// callers that have no way to hand the library a device workspace.
//
// paged_decode_attention needs scratch memory (the partition plan, the
// per-partition partial outputs and the status word) and asks its caller for
// it.  Some callers cannot provide that: a plain C host program with no device
// allocator of its own, a plugin or custom operator whose host framework owns
// every byte of device memory and offers no scratch, or a serving loop that
// must not call cudaMalloc once it is running (cudaMalloc can synchronise the
// device and may fail under a fixed memory budget).  For them this file keeps
// one fixed-size scratch array in the library's own device memory and runs the
// ordinary entry point on it.  Nothing here allocates.
#include <cuda_runtime.h>

#include "internal.h"
#include "pagedkv.h"

namespace {

// The scratch every call on a device shares.  Each GPU that loads the library
// holds it until the process exits.
static __device__ __align__(256) unsigned char g_static_scratch[PKV_STATIC_SCRATCH_BYTES];

// Device address of g_static_scratch in the current device's context.  In
// host code the array's name only stands in for the symbol; the address a
// kernel may use comes from cudaGetSymbolAddress with the device current.  It
// is looked up on every call rather than kept: a host-side lookup that
// allocates nothing, and one that stays right after cudaDeviceReset rebuilds
// the context (and with it the array) at a possibly different address.  The
// first lookup on a device loads the library's device code there, which is
// why that first call must come before any stream capture.
int scratch_on_current_device(void **out) {
  void *p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
  if (e != cudaSuccess || p == nullptr) {
    pkv::record_cuda_error(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
    return PKV_ECUDA;
  }
  *out = p;
  return PKV_OK;
}

// Largest partition count whose workspace fits the scratch, for a call that
// left the count to the library (num_splits == 0) but whose usual count, one
// partition per resident warp, needs more scratch than the array holds (FP8
// caches with more than 8 query rows per kv head at D = 128 keep 16-row
// partials, 16 KiB per partition).  The workspace size grows with the count,
// so a bisection over [1, 2^24] finds it; PKV_EWORKSPACE if even one
// partition does not fit.
int partitions_that_fit(int B, int Hq, int Hkv, int D, int cache_dtype, int q_dtype, int *splits) {
  const size_t cap = (size_t)PKV_STATIC_SCRATCH_BYTES;
  int lo = 0, hi = 1 << 24;  // need(lo) fits (lo > 0), need(hi + 1) does not
  while (lo < hi) {
    const int mid = lo + (hi - lo + 1) / 2;
    size_t need = 0;
    const int rc = paged_decode_workspace_bytes(B, Hq, Hkv, D, cache_dtype, q_dtype, mid, &need);
    if (rc != PKV_OK) return rc;
    if (need <= cap) lo = mid;
    else hi = mid - 1;
  }
  if (lo == 0) return PKV_EWORKSPACE;
  *splits = lo;
  return PKV_OK;
}

}  // namespace

extern "C" int paged_decode_attention_static(void *out, const void *q, int q_dtype, const void *k_cache,
                                             const void *v_cache, int cache_dtype, const float *k_scale,
                                             const float *v_scale, const int32_t *block_table,
                                             int max_blocks_per_seq, const int32_t *context_lens, int B,
                                             int Hq, int Hkv, int D, int64_t num_blocks, float scale,
                                             int num_splits, pkv_stream_t stream) {
  size_t need = 0;
  int rc = paged_decode_workspace_bytes(B, Hq, Hkv, D, cache_dtype, q_dtype, num_splits, &need);
  if (rc != PKV_OK) return rc;
  if (need > (size_t)PKV_STATIC_SCRATCH_BYTES) {
    if (num_splits != 0) return PKV_EWORKSPACE;  // the caller's own count, beyond the fixed capacity
    rc = partitions_that_fit(B, Hq, Hkv, D, cache_dtype, q_dtype, &num_splits);
    if (rc != PKV_OK) return rc;
  }
  void *scratch = nullptr;
  rc = scratch_on_current_device(&scratch);
  if (rc != PKV_OK) return rc;
  // Every byte the attention reads from its workspace is written earlier in the
  // same call, so the scratch needs no clearing between calls.
  return paged_decode_attention(out, q, q_dtype, k_cache, v_cache, cache_dtype, k_scale, v_scale, block_table,
                                max_blocks_per_seq, context_lens, B, Hq, Hkv, D, num_blocks, scale, num_splits,
                                scratch, (size_t)PKV_STATIC_SCRATCH_BYTES, stream);
}

extern "C" int paged_decode_static_status(pkv_stream_t stream, int *flags_out) {
  void *scratch = nullptr;
  const int rc = scratch_on_current_device(&scratch);
  if (rc != PKV_OK) return rc;
  return paged_decode_status(scratch, (size_t)PKV_STATIC_SCRATCH_BYTES, stream, flags_out);
}
