// api.cpp — the extern "C" boundary of libpagedkv.so: argument validation,
// kernel selection, TMA descriptor encoding, workspace layout and launches.
// Every check runs before the first launch, so a rejected call touches no
// memory.  No function here allocates device memory.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "pagedkv.h"
#include "mq_decode.h"
#include "prefill.h"

namespace pkv {

static thread_local int g_last_cuda_error = 0;

static int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return PKV_OK;
  g_last_cuda_error = static_cast<int>(e);
  return PKV_ECUDA;
}

void record_cuda_error(cudaError_t e) { g_last_cuda_error = static_cast<int>(e); }

static inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

WsLayout ws_layout(int B, int P, int D, int GC) {
  WsLayout L;
  size_t o = 0;
  L.hdr = o;
  o = align_up(o + sizeof(WsHeader), 256);
  L.prefix = o;
  o = align_up(o + sizeof(int32_t) * (size_t)(B + 1), 256);
  L.starts = o;
  o = align_up(o + sizeof(int4) * (size_t)(P + 1), 256);
  L.part_o = o;
  o = align_up(o + sizeof(float) * (size_t)P * 2 * GC * D, 256);
  L.part_lse = o;
  o = align_up(o + sizeof(float) * (size_t)P * 2 * GC, 256);
  L.cta_flags = o;
  o = align_up(o + sizeof(int32_t) * (size_t)P, 256);
  L.total = o;
  return L;
}

// ---------------------------------------------------------------------------
// Kernel registry and per-device facts.
// ---------------------------------------------------------------------------
namespace {

constexpr int kMaxKernels = 64;
constexpr int kMaxDevices = 64;

struct Registry {
  DecodeKernel k[kMaxKernels];
  int n = 0;
};

Registry &registry() {
  static Registry r;
  static std::once_flag once;
  std::call_once(once, [] {
    r.n += register_decode_bf16(r.k + r.n);
    r.n += register_decode_f16(r.k + r.n);
    r.n += register_decode_fp8(r.k + r.n);
    r.n += register_decode_f32(r.k + r.n);
  });
  return r;
}

// Route overrides set by pkv_set_route (PKV_ROUTE_AUTO = the rule of shapes).
std::atomic<int> g_route[2];

// Limit of every bounded in-kernel wait (a wait that runs out sets
// PKV_FLAG_TIMEOUT instead of hanging).
constexpr uint64_t kWaitLimitNs = 4000000000ull;

// Pending failure-path test requests (pkv_test_stall_next), one per kernel
// family, consumed by the next call that launches that family: the wait
// limit of that call, or 0.
std::atomic<uint64_t> g_stall[2];

// Sets the wait limit and the test hook of a launch from a pending request.
template <class Params>
void take_stall(Params &p, int which) {
  const uint64_t st = g_stall[which].exchange(0, std::memory_order_relaxed);
  p.stall_ns = st;
  p.timeout_ns = st ? st : kWaitLimitNs;
}

struct DeviceFacts {
  int sm_count = 0;
  int ctas_per_sm[kMaxKernels] = {};  // 0 = not yet configured
};
std::mutex g_dev_mu;
DeviceFacts g_dev[kMaxDevices];

// Configures kernel `ki` on the current device (opt-in shared memory) and
// returns its resident CTAs per SM and the SM count.
int kernel_occupancy(int ki, int *ctas_per_sm, int *sm_count) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_status(e);
  if (dev < 0 || dev >= kMaxDevices) return PKV_EUNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceFacts &f = g_dev[dev];
  if (f.sm_count == 0) {
    e = cudaDeviceGetAttribute(&f.sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_status(e);
  }
  if (f.ctas_per_sm[ki] == 0) {
    const DecodeKernel &k = registry().k[ki];
    e = cudaFuncSetAttribute(k.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)k.smem_bytes);
    if (e != cudaSuccess) return cuda_status(e);
    int nb = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, k.fn, k.warps * 32, k.smem_bytes);
    if (e != cudaSuccess) return cuda_status(e);
    if (nb <= 0) return PKV_EUNSUPPORTED;
    f.ctas_per_sm[ki] = nb;
  }
  *ctas_per_sm = f.ctas_per_sm[ki];
  *sm_count = f.sm_count;
  return PKV_OK;
}

// The current device's SM count (cached).
int device_sm_count(int *out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_status(e);
  if (dev < 0 || dev >= kMaxDevices) return PKV_EUNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceFacts &f = g_dev[dev];
  if (f.sm_count == 0) {
    e = cudaDeviceGetAttribute(&f.sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_status(e);
  }
  *out = f.sm_count;
  return PKV_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

int esize_of(int dtype) {
  switch (dtype) {
    case PKV_F32: return 4;
    case PKV_F16: return 2;
    case PKV_BF16: return 2;
    case PKV_FP8_E4M3: return 1;
  }
  return 0;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Tensor map over a [num_blocks][Hkv][16][D] cache as 2-D rows of 128 bytes
// wide boxes with the 128-byte swizzle; one box is 16 token rows x 128 bytes
// (or 8 lines of two 64-byte tokens).
int encode_cache_map(CUtensorMap *map, const void *base, int dtype, int64_t num_blocks, int Hkv, int D) {
  auto fn = encode_fn();
  if (!fn) return cuda_status(cudaErrorNotSupported);
  const int es = esize_of(dtype);
  const int rowb = D * es;
  cuuint64_t dims[2], strides[1];
  cuuint32_t box[2], estr[2] = {1, 1};
  const cuuint64_t tiles = (cuuint64_t)num_blocks * Hkv;
  if (rowb >= 128) {
    dims[0] = (cuuint64_t)D;
    dims[1] = tiles * kBlock;
    strides[0] = (cuuint64_t)rowb;
    box[0] = 128 / es;
    box[1] = kBlock;
  } else {
    dims[0] = 128 / es;
    dims[1] = tiles * kBlock * rowb / 128;
    strides[0] = 128;
    box[0] = 128 / es;
    box[1] = kBlock * rowb / 128;
  }
  const CUtensorMapDataType dt = es == 1   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : es == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16
                                           : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  CUresult r = fn(map, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cuda_status(cudaErrorInvalidValue);
  return PKV_OK;
}

// Encoded tensor maps of recently used caches.  A map depends only on the
// cache's base address, element type and dimensions, which make up the key,
// so a hit is always the map the encoder would produce; decode calls on the
// same cache (every layer step of a serving loop) skip the encoder.  Small
// and fixed in size, replaced round-robin; no allocation.
struct MapKey {
  const void *base;
  int64_t num_blocks;
  int dtype, Hkv, D;
  bool operator==(const MapKey &o) const {
    return base == o.base && num_blocks == o.num_blocks && dtype == o.dtype && Hkv == o.Hkv && D == o.D;
  }
};
struct MapCache {
  static constexpr int kEntries = 64;
  MapKey key[kEntries] = {};
  CUtensorMap map[kEntries];
  int used = 0, next = 0;
  std::mutex mu;
};
MapCache g_maps;

int cache_map(CUtensorMap *map, const void *base, int dtype, int64_t num_blocks, int Hkv, int D) {
  const MapKey k{base, num_blocks, dtype, Hkv, D};
  {
    std::lock_guard<std::mutex> lock(g_maps.mu);
    for (int i = 0; i < g_maps.used; ++i)
      if (g_maps.key[i] == k) {
        *map = g_maps.map[i];
        return PKV_OK;
      }
  }
  const int rc = encode_cache_map(map, base, dtype, num_blocks, Hkv, D);
  if (rc != PKV_OK) return rc;
  std::lock_guard<std::mutex> lock(g_maps.mu);
  const int slot = g_maps.used < MapCache::kEntries ? g_maps.used++ : g_maps.next;
  if (g_maps.used == MapCache::kEntries) g_maps.next = (slot + 1) % MapCache::kEntries;
  g_maps.key[slot] = k;
  g_maps.map[slot] = *map;
  return PKV_OK;
}

struct Choice {
  int ki;   // registry index
  int GC;   // query rows per unit
  int NC;   // units per kv head
};

// Picks the kernel for a shape: tensor cores (8-row units, unused columns
// padded; 16-row units on fp8 caches past 8 rows) for every group size on
// 16-bit and fp8 caches — even for
// MHA the mma.sync block step measured faster on GB300 than the CUDA-core one
// (5.83 vs 5.56 TB/s, fp16 MHA layer) — and CUDA cores for fp32 caches.  The
// first compiled match is the default pipeline shape.  A build with
// PKV_SWEEP_SHAPES defined (pipeline-shape sweeps, not the product build)
// also compiles alternative shapes and lets PKV_PATH=mma|simt,
// PKV_DECODE_WARPS, PKV_DECODE_STAGES and PKV_DECODE_GC=8 in the environment
// pick among them.
int choose_kernel(int cache_dtype, int q_dtype, int D, int R, Choice *c) {
#ifdef PKV_SWEEP_SHAPES
  static const int force = [] {
    const char *v = std::getenv("PKV_PATH");
    if (v && std::strcmp(v, "simt") == 0) return 1;
    if (v && std::strcmp(v, "mma") == 0) return 2;
    return 0;
  }();
  static const int want_warps = [] {
    const char *v = std::getenv("PKV_DECODE_WARPS");
    return v ? std::atoi(v) : 0;
  }();
  static const int want_stages = [] {
    const char *v = std::getenv("PKV_DECODE_STAGES");
    return v ? std::atoi(v) : 0;
  }();
  static const int want_gc = [] {
    const char *v = std::getenv("PKV_DECODE_GC");
    return v ? std::atoi(v) : 0;
  }();
#else
  constexpr int force = 0, want_warps = 0, want_stages = 0, want_gc = 0;
#endif
  const bool mma = cache_dtype != PKV_F32 && force != 1;
  // fp8 caches serve a kv head with more than 8 rows in 16-row units: each
  // E4M3 element is widened once per 16 rows instead of once per 8 (on the
  // 32K fp8 layer at 16 rows, one 16-row unit per kv head against two 8-row
  // units streaming the same blocks)
  int GC = mma ? 8 : (R >= 2 ? 2 : 1);
  if (mma && cache_dtype == PKV_FP8_E4M3 && R > 8 && want_gc != 8) GC = 16;
  Registry &r = registry();
  int first = -1;
  for (int pass = 0; pass < 2 && first < 0; ++pass) {
    if (pass == 1) {
      if (GC != 16) break;
      GC = 8;  // no 16-row kernel for this (q dtype, D): 8-row units
    }
    for (int i = 0; i < r.n; ++i) {
      const DecodeKernel &k = r.k[i];
      if (k.mma == (mma ? 1 : 0) && k.cache_dtype == cache_dtype && k.q_dtype == q_dtype && k.D == D && k.GC == GC) {
        if (first < 0) first = i;
        if ((want_warps == 0 || k.warps == want_warps) && (want_stages == 0 || k.stages == want_stages)) {
          first = i;
          break;
        }
      }
    }
  }
  if (first < 0) return PKV_EUNSUPPORTED;
  c->ki = first;
  c->GC = GC;
  c->NC = (R + GC - 1) / GC;
  return PKV_OK;
}

int validate_decode_shapes(int q_dtype, int cache_dtype, int B, int q_len, int Hq, int Hkv, int D,
                           int64_t num_blocks, int max_blocks) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || num_blocks <= 0 || max_blocks <= 0) return PKV_EINVAL;
  if (q_len < 1 || q_len > PKV_MAX_Q_LEN) return PKV_EINVAL;
  if (max_blocks > (1 << 26)) return PKV_EUNSUPPORTED;  // 16 * max_blocks stays below 2^30
  if (Hq % Hkv != 0) return PKV_EINVAL;
  if (esize_of(cache_dtype) == 0 || esize_of(q_dtype) == 0 || q_dtype == PKV_FP8_E4M3) return PKV_EINVAL;
  if (D != 64 && D != 128) return PKV_EUNSUPPORTED;
  if (cache_dtype == PKV_F32 && q_dtype != PKV_F32) return PKV_EUNSUPPORTED;
  if ((cache_dtype == PKV_F16 || cache_dtype == PKV_BF16) && q_dtype != cache_dtype) return PKV_EUNSUPPORTED;
  if (cache_dtype == PKV_FP8_E4M3 && q_dtype == PKV_F32) return PKV_EUNSUPPORTED;
  // TMA row coordinates and the work-item count are 32-bit
  if ((double)num_blocks * Hkv * kBlock >= 2147483000.0) return PKV_EUNSUPPORTED;
  const int R = q_len * (Hq / Hkv);  // query rows per kv head; units per kv head <= R
  if ((double)B * max_blocks * Hkv * R >= 2147483000.0) return PKV_EUNSUPPORTED;
  return PKV_OK;
}

// Resolves the kernel and the partition count for a call.
int plan_call(int cache_dtype, int q_dtype, int B, int q_len, int Hq, int Hkv, int D, int num_splits, Choice *c,
              int *P) {
  int rc = choose_kernel(cache_dtype, q_dtype, D, q_len * (Hq / Hkv), c);
  if (rc != PKV_OK) return rc;
  if (num_splits < 0) return PKV_EINVAL;
  if (num_splits > 0) {
    *P = num_splits;
  } else {
    int ctas = 0, sms = 0;
    rc = kernel_occupancy(c->ki, &ctas, &sms);
    if (rc != PKV_OK) return rc;
    *P = sms * ctas * registry().k[c->ki].warps;
  }
  if (*P > (1 << 24)) return PKV_EINVAL;
  (void)B;
  return PKV_OK;
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" {

int pkv_version(void) { return 10100; }

int pkv_set_route(int which, int choice) {
  if (which == PKV_ROUTE_MULTI_QUERY) {
    if (choice < PKV_ROUTE_AUTO || choice > PKV_MQ_UNITS) return PKV_EINVAL;
  } else if (which == PKV_ROUTE_PREFILL) {
    if (choice < PKV_ROUTE_AUTO || choice > PKV_PREFILL_PER_ITEM) return PKV_EINVAL;
  } else {
    return PKV_EINVAL;
  }
  g_route[which].store(choice, std::memory_order_relaxed);
  return PKV_OK;
}

int pkv_test_stall_next(int which, uint64_t limit_ns) {
  if (which != PKV_STALL_DECODE && which != PKV_STALL_PREFILL) return PKV_EINVAL;
  if (limit_ns != 0 && (limit_ns < 1000000ull || limit_ns > 10000000000ull)) return PKV_EINVAL;
  g_stall[which].store(limit_ns, std::memory_order_relaxed);
  return PKV_OK;
}

int pkv_get_route(int which) {
  if (which != PKV_ROUTE_MULTI_QUERY && which != PKV_ROUTE_PREFILL) return PKV_EINVAL;
  return g_route[which].load(std::memory_order_relaxed);
}

int pkv_last_cuda_error(void) { return g_last_cuda_error; }

const char *pkv_status_string(int status) {
  switch (status) {
    case PKV_OK: return "ok";
    case PKV_EINVAL: return "invalid argument";
    case PKV_EUNSUPPORTED: return "unsupported shape or dtype combination";
    case PKV_EWORKSPACE: return "workspace missing, misaligned or too small";
    case PKV_ECUDA: return "CUDA runtime error";
    case PKV_ETIMEOUT: return "an in-kernel wait timed out";
    case PKV_EOOM: return "no free physical block";
    case PKV_ERANGE: return "value out of range";
    case PKV_ENOTFOUND: return "unknown sequence id";
  }
  return "unknown status";
}

int paged_kv_append(const void *k_new, const void *v_new, int new_dtype, void *k_cache, void *v_cache,
                    int cache_dtype, float *k_scale, float *v_scale, const int64_t *slot_mapping, int B, int Hkv,
                    int D, int64_t num_blocks, pkv_stream_t stream) {
  if (B < 0 || Hkv <= 0 || num_blocks <= 0) return PKV_EINVAL;
  if (esize_of(cache_dtype) == 0 || esize_of(new_dtype) == 0) return PKV_EINVAL;
  if (D != 64 && D != 128) return PKV_EUNSUPPORTED;
  if (B == 0) return PKV_OK;
  if (!k_new || !v_new || !k_cache || !v_cache || !slot_mapping) return PKV_EINVAL;
  if (cache_dtype == PKV_FP8_E4M3) {
    if (new_dtype == PKV_FP8_E4M3) return PKV_EUNSUPPORTED;
    if (!k_scale || !v_scale) return PKV_EINVAL;
  } else {
    if (new_dtype != cache_dtype) return PKV_EUNSUPPORTED;
    if (!aligned16(k_new) || !aligned16(v_new)) return PKV_EINVAL;
  }
  if (!aligned16(k_cache) || !aligned16(v_cache)) return PKV_EINVAL;
  return cuda_status(launch_append(k_new, v_new, new_dtype, k_cache, v_cache, cache_dtype, k_scale, v_scale,
                                   slot_mapping, B, Hkv, D, num_blocks, reinterpret_cast<cudaStream_t>(stream)));
}

int paged_decode_multi_workspace_bytes(int B, int q_len, int Hq, int Hkv, int D, int cache_dtype, int q_dtype,
                                       int num_splits, size_t *bytes_out) {
  if (!bytes_out) return PKV_EINVAL;
  int rc = validate_decode_shapes(q_dtype, cache_dtype, B, q_len, Hq, Hkv, D, 1, 1);
  if (rc != PKV_OK) return rc;
  Choice c;
  int P = 0;
  rc = plan_call(cache_dtype, q_dtype, B, q_len, Hq, Hkv, D, num_splits, &c, &P);
  if (rc != PKV_OK) return rc;
  size_t total = ws_layout(B, P, D, c.GC).total;
  if (q_len >= 2 && num_splits == 0 && D == kMqHeadDim && q_len * (Hq / Hkv) <= kMqRows && B <= kMqMaxBatch &&
      (cache_dtype == PKV_BF16 || cache_dtype == PKV_F16 ||
       (cache_dtype == PKV_FP8_E4M3 && q_len * (Hq / Hkv) <= kMqRowsFp8))) {
    int sms = 0;
    rc = device_sm_count(&sms);
    if (rc != PKV_OK) return rc;
    const size_t mq = mq_ws_layout(B, sms).total;  // the transposed kernel's partials
    if (mq > total) total = mq;
  }
  *bytes_out = total;
  return PKV_OK;
}

int paged_kv_append_calibrated(const void *k_new, const void *v_new, int new_dtype, void *k_cache, void *v_cache,
                               int cache_dtype, float *k_scale, float *v_scale, const int64_t *slot_mapping, int B,
                               int Hkv, int D, int64_t num_blocks, pkv_stream_t stream) {
  if (cache_dtype != PKV_FP8_E4M3)
    return paged_kv_append(k_new, v_new, new_dtype, k_cache, v_cache, cache_dtype, k_scale, v_scale, slot_mapping, B,
                           Hkv, D, num_blocks, stream);
  if (B < 0 || Hkv <= 0 || num_blocks <= 0) return PKV_EINVAL;
  if (esize_of(new_dtype) == 0) return PKV_EINVAL;
  if (new_dtype == PKV_FP8_E4M3) return PKV_EUNSUPPORTED;
  if (D != 64 && D != 128) return PKV_EUNSUPPORTED;
  if (B == 0) return PKV_OK;
  if (!k_new || !v_new || !k_cache || !v_cache || !slot_mapping || !k_scale || !v_scale) return PKV_EINVAL;
  if (!aligned16(k_cache) || !aligned16(v_cache)) return PKV_EINVAL;
  return cuda_status(launch_append_calibrated(k_new, v_new, new_dtype, k_cache, v_cache, k_scale, v_scale,
                                              slot_mapping, B, Hkv, D, num_blocks,
                                              reinterpret_cast<cudaStream_t>(stream)));
}

int paged_decode_workspace_bytes(int B, int Hq, int Hkv, int D, int cache_dtype, int q_dtype, int num_splits,
                                 size_t *bytes_out) {
  return paged_decode_multi_workspace_bytes(B, 1, Hq, Hkv, D, cache_dtype, q_dtype, num_splits, bytes_out);
}

int paged_decode_attention(void *out, const void *q, int q_dtype, const void *k_cache, const void *v_cache,
                           int cache_dtype, const float *k_scale, const float *v_scale, const int32_t *block_table,
                           int max_blocks_per_seq, const int32_t *context_lens, int B, int Hq, int Hkv, int D,
                           int64_t num_blocks, float scale, int num_splits, void *workspace, size_t workspace_bytes,
                           pkv_stream_t stream) {
  return paged_decode_attention_multi(out, q, q_dtype, k_cache, v_cache, cache_dtype, k_scale, v_scale, block_table,
                                      max_blocks_per_seq, context_lens, B, 1, 0, Hq, Hkv, D, num_blocks, scale,
                                      num_splits, workspace, workspace_bytes, stream);
}

// The two prefill kernels run one tile pipeline and differ in scheduling.
// One CTA per work item (row tile x kv head x sequence) runs the per-tile
// loop fastest and suits long items: new tokens after a cached prefix of
// thousands of positions.  The persistent kernel (one CTA per SM walking its
// items) saves each item's start-up and balances short items of unequal
// length: prompts without a long prefix.  The longest context the block
// table can describe (max_blocks * block size) less the new tokens bounds
// the prefix; a bound of 2048 positions or more picks one CTA per item, or
// 1024 for items of at most 64 rows (a few new tokens of one group), which
// that kernel serves with row replicas (measured on 70B-layer shapes: at
// 1024 positions the two kernels tie, at 1500 one CTA per item is 11 %
// faster, at 300-512 the persistent kernel is 14-15 % faster).
// pkv_set_route(PKV_ROUTE_PREFILL, ...) overrides the choice.
static cudaError_t launch_prefill_auto(const PrefillParams &p, int cache_dtype, const CUtensorMap &tmK,
                                       const CUtensorMap &tmV, cudaStream_t s) {
  const int64_t bound = (int64_t)p.max_q_len * p.G <= 64 ? 1024 : 2048;
  bool tiles = (int64_t)p.max_blocks * kBlock - p.max_q_len >= bound;
  const int force = g_route[PKV_ROUTE_PREFILL].load(std::memory_order_relaxed);
  if (force == PKV_PREFILL_PER_ITEM) tiles = true;
  if (force == PKV_PREFILL_PERSISTENT) tiles = false;
  return tiles ? launch_prefill_tiles(p, cache_dtype, tmK, tmV, s) : launch_prefill(p, cache_dtype, tmK, tmV, s);
}

int paged_decode_attention_multi(void *out, const void *q, int q_dtype, const void *k_cache, const void *v_cache,
                                 int cache_dtype, const float *k_scale, const float *v_scale,
                                 const int32_t *block_table, int max_blocks_per_seq, const int32_t *context_lens,
                                 int B, int q_len, int window, int Hq, int Hkv, int D, int64_t num_blocks,
                                 float scale, int num_splits, void *workspace, size_t workspace_bytes,
                                 pkv_stream_t stream) {
  int rc = validate_decode_shapes(q_dtype, cache_dtype, B, q_len, Hq, Hkv, D, num_blocks, max_blocks_per_seq);
  if (rc != PKV_OK) return rc;
  if (window < 0) return PKV_EINVAL;
  if (!std::isfinite(scale)) return PKV_EINVAL;
  if (B == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache || !block_table || !context_lens) return PKV_EINVAL;
  if (cache_dtype == PKV_FP8_E4M3 && (!k_scale || !v_scale)) return PKV_EINVAL;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache)) return PKV_EINVAL;
  Choice c;
  int P = 0;
  rc = plan_call(cache_dtype, q_dtype, B, q_len, Hq, Hkv, D, num_splits, &c, &P);
  if (rc != PKV_OK) return rc;
  const WsLayout L = ws_layout(B, P, D, c.GC);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < L.total)
    return PKV_EWORKSPACE;
  if (q_len >= 2 && num_splits == 0) {
    // Several new tokens per sequence on a 16-bit cache: a tensor-core
    // kernel streams each (sequence, kv head)'s K/V once for all of its
    // q_len * G rows (the decode kernel's units below stream it once per
    // unit).
    //  * up to 32 rows and head dim 128: the transposed kernel (positions on
    //    the tensor core's M side, stream-K over every item's tiles, so any
    //    batch fills the GPU);
    //  * otherwise the prefill kernel with 128-row tiles, when its grid of
    //    (sequence, kv head, row tile) items fills the GPU (no context split;
    //    on the 70B layer at 64 rows it is faster than the transposed kernel,
    //    whose softmax work grows with the rows);
    //  * the transposed kernel for 33-64 rows on grids the prefill kernel
    //    cannot fill.
    // pkv_set_route(PKV_ROUTE_MULTI_QUERY, ...) forces one route where it
    // applies (for measurement and tests).
    int sms = 0;
    rc = device_sm_count(&sms);
    if (rc != PKV_OK) return rc;
    const int force = g_route[PKV_ROUTE_MULTI_QUERY].load(std::memory_order_relaxed);
    const bool units = force == PKV_MQ_UNITS;
    const bool no_mq = units || force == PKV_MQ_PREFILL;
    const bool want_mq = force == PKV_MQ_TRANSPOSED;
    const int G = Hq / Hkv;
    const int R = q_len * G;
    const int64_t tiles = ((int64_t)q_len * G + 127) / 128;
    const bool prefill_fills = (int64_t)B * Hkv * tiles >= sms && B <= 65535;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // FP8 caches take the decode kernel's units (16 rows each past 8 rows):
    // the transposed kernel widens each tile to f16 in shared memory, which
    // on 32 KiB fp8 tiles costs more than the tile's HBM time (~2.1 TB/s
    // whatever the rows, against the units' 6.1 / 4.6 / 2.4 TB/s at 8 / 16 /
    // 32 rows on the 32K fp8 layer); it runs only when forced.  FP8 caches
    // have no prefill route.
    const bool fp8 = cache_dtype == PKV_FP8_E4M3;
    const bool fp8_mq = fp8 && R <= kMqRowsFp8 && want_mq;
    if (!no_mq && (cache_dtype == PKV_BF16 || cache_dtype == PKV_F16 || fp8_mq) && scale > 0.f &&
        D == kMqHeadDim && R <= kMqRows && B <= kMqMaxBatch && (R <= 32 || !prefill_fills || want_mq)) {
      const MqWsLayout M = mq_ws_layout(B, sms);
      if (workspace_bytes >= M.total) {
        CUtensorMap tmK, tmV;
        rc = cache_map(&tmK, k_cache, cache_dtype, num_blocks, Hkv, D);
        if (rc != PKV_OK) return rc;
        rc = cache_map(&tmV, v_cache, cache_dtype, num_blocks, Hkv, D);
        if (rc != PKV_OK) return rc;
        uint8_t *ws = static_cast<uint8_t *>(workspace);
        MqParams mp;
        std::memset(&mp, 0, sizeof(mp));
        mp.out = out;
        mp.q = q;
        mp.k_scale = k_scale;
        mp.v_scale = v_scale;
        mp.block_table = block_table;
        mp.context_lens = context_lens;
        mp.status = &reinterpret_cast<WsHeader *>(ws)->status;
        mp.cta_flags = reinterpret_cast<int32_t *>(ws + M.cta_flags);
        mp.prefix = reinterpret_cast<int32_t *>(ws + M.prefix);
        mp.part_o = reinterpret_cast<float *>(ws + M.part_o);
        mp.part_lse = reinterpret_cast<float *>(ws + M.part_lse);
        mp.num_blocks = num_blocks;
        mp.B = B;
        mp.q_len = q_len;
        mp.Hq = Hq;
        mp.Hkv = Hkv;
        mp.G = G;
        mp.R = R;
        mp.max_blocks = max_blocks_per_seq;
        mp.window = window < (1 << 30) ? window : 0;
        mp.scale_log2 = scale * 1.4426950408889634f;
        mp.timeout_ns = kWaitLimitNs;
        return cuda_status(launch_mq_decode(mp, cache_dtype, q_dtype, tmK, tmV, sms, s));
      }
    }
    if (!units && (cache_dtype == PKV_BF16 || cache_dtype == PKV_F16) && scale > 0.f && prefill_fills) {
      CUtensorMap tmK, tmV;
      rc = cache_map(&tmK, k_cache, cache_dtype, num_blocks, Hkv, D);
      if (rc != PKV_OK) return rc;
      rc = cache_map(&tmV, v_cache, cache_dtype, num_blocks, Hkv, D);
      if (rc != PKV_OK) return rc;
      WsHeader *hdr = reinterpret_cast<WsHeader *>(static_cast<uint8_t *>(workspace) + L.hdr);
      cudaError_t e = cudaMemsetAsync(&hdr->status, 0, sizeof(int32_t), s);
      if (e != cudaSuccess) return cuda_status(e);
      PrefillParams pp;
      std::memset(&pp, 0, sizeof(pp));
      pp.out = out;
      pp.q = q;
      pp.block_table = block_table;
      pp.context_lens = context_lens;
      pp.q_start = nullptr;
      pp.uniform_q_len = q_len;
      pp.status = &hdr->status;
      pp.num_blocks = num_blocks;
      pp.B = B;
      pp.Hq = Hq;
      pp.Hkv = Hkv;
      pp.D = D;
      pp.G = G;
      pp.max_blocks = max_blocks_per_seq;
      pp.max_q_len = q_len;
      pp.max_tiles = (int)tiles;
      pp.window = window < (1 << 30) ? window : 0;
      pp.scale_log2 = scale * 1.4426950408889634f;
      take_stall(pp, PKV_STALL_PREFILL);
      return cuda_status(launch_prefill_auto(pp, cache_dtype, tmK, tmV, s));
    }
  }
  const DecodeKernel &k = registry().k[c.ki];
  int ctas = 0, sms = 0;
  rc = kernel_occupancy(c.ki, &ctas, &sms);  // also opts the kernel into its shared memory
  if (rc != PKV_OK) return rc;

  CUtensorMap tmK, tmV;
  rc = cache_map(&tmK, k_cache, cache_dtype, num_blocks, Hkv, D);
  if (rc != PKV_OK) return rc;
  rc = cache_map(&tmV, v_cache, cache_dtype, num_blocks, Hkv, D);
  if (rc != PKV_OK) return rc;

  uint8_t *ws = static_cast<uint8_t *>(workspace);
  DecodeParams p;
  std::memset(&p, 0, sizeof(p));
  p.out = out;
  p.q = q;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.block_table = block_table;
  p.context_lens = context_lens;
  p.hdr = reinterpret_cast<WsHeader *>(ws + L.hdr);
  p.prefix = reinterpret_cast<int32_t *>(ws + L.prefix);
  p.starts = reinterpret_cast<int4 *>(ws + L.starts);
  p.part_o = reinterpret_cast<float *>(ws + L.part_o);
  p.part_lse = reinterpret_cast<float *>(ws + L.part_lse);
  p.cta_flags = reinterpret_cast<int32_t *>(ws + L.cta_flags);
  p.num_blocks = num_blocks;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.D = D;
  p.G = Hq / Hkv;
  p.GC = c.GC;
  p.NC = c.NC;
  p.HU = Hkv * c.NC;
  p.q_len = q_len;
  p.R = q_len * p.G;
  // a window of 2^30 positions or more covers any context this call accepts
  p.window = window < (1 << 30) ? window : 0;
  p.wlen = p.window > 0 ? p.window : (1 << 30);
  p.P = P;
  p.max_blocks = max_blocks_per_seq;
  p.out_dtype = q_dtype;
  p.scale_log2 = scale * 1.4426950408889634f;
  take_stall(p, PKV_STALL_DECODE);

  p.inline_plan = B + 1 <= kInlinePrefix ? 1 : 0;
  p.n_ctas = (P + k.warps - 1) / k.warps;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool pdl = s != nullptr;  // programmatic launch on explicit streams only
  cudaError_t e = cudaSuccess;
  if (!p.inline_plan) {
    e = launch_plan(p, s);
    if (e != cudaSuccess) return cuda_status(e);
  }

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.n_ctas);
  cfg.blockDim = dim3(k.warps * 32);
  cfg.dynamicSmemBytes = k.smem_bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  void *args[3] = {&p, &tmK, &tmV};
  e = cudaLaunchKernelExC(&cfg, k.fn, args);
  if (e != cudaSuccess) return cuda_status(e);
  e = launch_splitk_merge(p, s, pdl);
  return cuda_status(e);
}

int paged_prefill_attention(void *out, const void *q, int q_dtype, const void *k_cache, const void *v_cache,
                            int cache_dtype, const int32_t *block_table, int max_blocks_per_seq,
                            const int32_t *context_lens, const int32_t *q_start, int B, int max_q_len, int Hq,
                            int Hkv, int D, int64_t num_blocks, float scale, int window, int32_t *status,
                            pkv_stream_t stream) {
  int rc = validate_decode_shapes(q_dtype, cache_dtype, B, 1, Hq, Hkv, D, num_blocks, max_blocks_per_seq);
  if (rc != PKV_OK) return rc;
  if (cache_dtype != PKV_F16 && cache_dtype != PKV_BF16) return PKV_EUNSUPPORTED;
  if (!(scale > 0.f) || !std::isfinite(scale) || window < 0 || max_q_len < 0) return PKV_EINVAL;
  if (B > 65535 || Hkv > 65535) return PKV_EUNSUPPORTED;
  const int G = Hq / Hkv;
  const int64_t tiles = ((int64_t)max_q_len * G + 127) / 128;
  if (tiles > INT32_MAX) return PKV_EUNSUPPORTED;
  if (B == 0 || tiles == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache || !block_table || !context_lens || !q_start) return PKV_EINVAL;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache)) return PKV_EINVAL;
  CUtensorMap tmK, tmV;
  rc = cache_map(&tmK, k_cache, cache_dtype, num_blocks, Hkv, D);
  if (rc != PKV_OK) return rc;
  rc = cache_map(&tmV, v_cache, cache_dtype, num_blocks, Hkv, D);
  if (rc != PKV_OK) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (status) {
    cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int32_t), s);
    if (e != cudaSuccess) return cuda_status(e);
  }
  PrefillParams p;
  std::memset(&p, 0, sizeof(p));
  p.out = out;
  p.q = q;
  p.block_table = block_table;
  p.context_lens = context_lens;
  p.q_start = q_start;
  p.status = status;
  p.num_blocks = num_blocks;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.D = D;
  p.G = G;
  p.max_blocks = max_blocks_per_seq;
  p.max_q_len = max_q_len;
  p.max_tiles = (int)tiles;
  p.window = window < (1 << 30) ? window : 0;
  p.scale_log2 = scale * 1.4426950408889634f;
  take_stall(p, PKV_STALL_PREFILL);
  return cuda_status(launch_prefill_auto(p, cache_dtype, tmK, tmV, s));
}

int paged_decode_status(const void *workspace, size_t workspace_bytes, pkv_stream_t stream, int *flags_out) {
  if (!workspace || workspace_bytes < sizeof(WsHeader)) return PKV_EWORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t status = 0;
  cudaError_t e = cudaMemcpyAsync(&status, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_status(e);
  if (flags_out) *flags_out = status;
  if (status & PKV_FLAG_TIMEOUT) return PKV_ETIMEOUT;
  if (status & (PKV_FLAG_BAD_LEN | PKV_FLAG_BAD_BLOCK | PKV_FLAG_RANGE)) return PKV_ERANGE;
  return PKV_OK;
}

int paged_decode_merge(void *out, int out_dtype, const float *o_partial, const float *lse, int B, int Hq, int D,
                       int S, pkv_stream_t stream) {
  if (B < 0 || Hq <= 0 || D <= 0 || S <= 0) return PKV_EINVAL;
  if (out_dtype != PKV_F32 && out_dtype != PKV_F16 && out_dtype != PKV_BF16) return PKV_EINVAL;
  if (B == 0) return PKV_OK;
  if (!out || !o_partial || !lse) return PKV_EINVAL;
  return cuda_status(launch_merge(out, out_dtype, o_partial, lse, B, Hq, D, S, reinterpret_cast<cudaStream_t>(stream)));
}

int paged_kv_copy_blocks(void *k_cache, void *v_cache, int cache_dtype, float *k_scale, float *v_scale,
                         const int32_t *src_dst_pairs, int n_pairs, int Hkv, int D, int64_t num_blocks,
                         pkv_stream_t stream) {
  if (n_pairs < 0 || Hkv <= 0 || num_blocks <= 0) return PKV_EINVAL;
  if (esize_of(cache_dtype) == 0) return PKV_EINVAL;
  if (D != 64 && D != 128) return PKV_EUNSUPPORTED;
  if (n_pairs == 0) return PKV_OK;
  if (!k_cache || !v_cache || !src_dst_pairs) return PKV_EINVAL;
  if (cache_dtype == PKV_FP8_E4M3 && (!k_scale || !v_scale)) return PKV_EINVAL;
  if (!aligned16(k_cache) || !aligned16(v_cache)) return PKV_EINVAL;
  return cuda_status(launch_copy_blocks(k_cache, v_cache, cache_dtype, k_scale, v_scale, src_dst_pairs, n_pairs,
                                        Hkv, D, num_blocks, reinterpret_cast<cudaStream_t>(stream)));
}

int pkv_copy(void *dst, const void *src, size_t bytes, pkv_stream_t stream) {
  if (bytes == 0) return PKV_OK;
  if (!dst || !src || (bytes & 15u) != 0 || !aligned16(dst) || !aligned16(src)) return PKV_EINVAL;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_status(e);
  return cuda_status(launch_copy(dst, src, bytes, sms, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
