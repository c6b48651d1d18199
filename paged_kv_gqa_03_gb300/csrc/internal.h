// internal.h — declarations shared by the C-ABI layer (api.cpp) and the kernel
// translation units.  Not part of the public interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace pkv {

constexpr int kBlock = 16;      // tokens per physical block (PKV_BLOCK_SIZE)
constexpr int kChunkMax = 16;   // most query rows one work unit serves

// Workspace header written by the plan kernel each call.
// Workspace header.  `status` is published by the merge kernel at the end of
// every call: the OR of the plan's flags (when the plan kernel ran) and of
// every decode CTA's flags.
struct WsHeader {
  int32_t status;      // PKV_FLAG_* bits of the last call
  int32_t plan_flags;  // written by the plan kernel
  int32_t P;           // partitions (warp workers)
  int32_t W;           // total (unit, block) work items
  int32_t B;
  int32_t HU;          // units per sequence = Hkv * NC
  int32_t pad[58];     // 256 bytes
};

// Batches up to this size are planned inside the decode kernel (each CTA
// scans context_lens into shared memory); larger ones use the plan kernel.
constexpr int kInlinePrefix = 2048;

// Per stage of a warp's pipeline: what the producer issued into it (one
// block, or two consecutive blocks of one unit on the two-block fp8 path).
struct StageMeta {
  int32_t b, hu, j, nvalid;  // nvalid = min(16, rem): cache rows of the block inside ctx
  float ks, vs;              // fp8 scales of the (first) block
  int32_t flags;
  int32_t rem;               // ctx - 16 j: positions of the sequence from this block on
  float ks1, vs1;            // fp8 scales of the second block
  int32_t nb;                // blocks in the stage (1 or 2)
  int32_t pad;
};
enum : int32_t {
  kFirst = 1,     // first block of a segment: reset state, load q
  kLast = 2,      // last block of a segment: finalise
  kComplete = 4,  // the segment is the whole unit: write the output directly
  kWFirst = 8,    // the segment is its worker's first (partial slot 0, else 1)
};

struct DecodeParams {
  void *out;
  const void *q;
  const float *k_scale;
  const float *v_scale;
  const int32_t *block_table;
  const int32_t *context_lens;
  WsHeader *hdr;
  int32_t *prefix;      // [B+1] exclusive prefix of blocks per sequence
  int4 *starts;         // [P+1] {s, b, hu, j} of each worker's first item
  float *part_o;        // [P][2][GC][D]
  float *part_lse;      // [P][2][GC], log2 domain
  int32_t *cta_flags;   // [decode CTAs] PKV_FLAG_* bits of each decode CTA
  int64_t num_blocks;
  int B, Hq, Hkv, D, G, GC, NC, HU, P;
  int q_len;            // new query tokens per sequence (1 = plain decode)
  int R;                // query rows per kv head = q_len * G, cut into NC chunks of GC
  int window;           // sliding window W (0 = none): a row sees [lim - W, lim)
  int wlen;             // W, or 1 << 30 without a window (visible-range width)
  int max_blocks;
  int out_dtype;
  float scale_log2;     // softmax scale * log2(e)
  uint64_t timeout_ns;
  uint64_t stall_ns;    // failure-path test hook (pkv_test_stall_next): 0 = off
  int inline_plan;      // 1: the decode kernel computes prefix and partition starts itself
  int n_ctas;           // decode grid size
};

#ifdef __CUDACC__
// Context length clamped to [0, 16 * max_blocks].
__device__ __forceinline__ int clamped_len(const DecodeParams &p, int ctx) {
  return ctx < 0 ? 0 : (ctx > p.max_blocks * kBlock ? p.max_blocks * kBlock : ctx);
}
// First block any row of a sequence of (clamped) length ctx can see: with a
// window, row 0's window starts at ctx - (q_len - 1) - W.
__device__ __forceinline__ int first_block(const DecodeParams &p, int ctx) {
  const int lo = p.window > 0 ? ctx - (p.q_len - 1) - p.window : 0;
  return lo > 0 ? lo / kBlock : 0;
}
// Work items (blocks streamed per unit) of a sequence of (clamped) length ctx.
__device__ __forceinline__ int seq_items(const DecodeParams &p, int ctx) {
  return (ctx + kBlock - 1) / kBlock - first_block(p, ctx);
}
// Partitions that receive work: P, or one per work item when the call has
// fewer items than partitions (a small step: more partitions would only add
// empty ranges for the merge to walk).  Partition w < Pe covers items
// [W w / Pe, W (w + 1) / Pe); the decode kernel, the plan and the merge
// compute it alike from W.
__device__ __forceinline__ int64_t active_partitions(const DecodeParams &p, int64_t W) {
  return W < p.P ? (W > 0 ? W : 1) : p.P;
}
#endif

// Records a CUDA error for pkv_last_cuda_error() on the calling thread.
void record_cuda_error(cudaError_t e);

struct WsLayout {
  size_t hdr, prefix, starts, part_o, part_lse, cta_flags, total;
};
WsLayout ws_layout(int B, int P, int D, int GC);  // GC = rows per unit

// One compiled decode kernel variant.
struct DecodeKernel {
  const void *fn;       // __global__ void (DecodeParams, CUtensorMap, CUtensorMap)
  int mma;              // 1 = tensor-core (mma.sync) path, 0 = CUDA-core path
  int cache_dtype, q_dtype, D, GC;
  int warps, stages;
  size_t smem_bytes;
};
// Appends the variants a translation unit compiled; returns how many.
int register_decode_bf16(DecodeKernel *out);
int register_decode_f16(DecodeKernel *out);
int register_decode_fp8(DecodeKernel *out);
int register_decode_f32(DecodeKernel *out);

// Paged prefill (tcgen05): each sequence's new tokens attend causally.
struct PrefillParams {
  void *out;
  const void *q;
  const int32_t *block_table;
  const int32_t *context_lens;
  const int32_t *q_start;   // [B+1] row offsets of each sequence's new tokens in q / out,
                            // or null: every sequence has uniform_q_len new tokens
  int uniform_q_len;
  int32_t *status;          // PKV_FLAG_* bits (may be null)
  int64_t num_blocks;
  int B, Hq, Hkv, D, G, max_blocks, max_q_len, max_tiles;
  int window;               // 0 = none
  float scale_log2;         // softmax scale * log2(e), > 0
  uint64_t timeout_ns;
  uint64_t stall_ns;        // failure-path test hook (pkv_test_stall_next): 0 = off
};
// Launches the prefill kernel for (cache dtype, D); cudaErrorNotSupported for
// a combination that is not compiled.
cudaError_t launch_prefill(const PrefillParams &p, int cache_dtype, const CUtensorMap &tmK, const CUtensorMap &tmV,
                           cudaStream_t stream);

cudaError_t launch_plan(const DecodeParams &p, cudaStream_t stream);
cudaError_t launch_splitk_merge(const DecodeParams &p, cudaStream_t stream, bool pdl);
cudaError_t launch_merge(void *out, int out_dtype, const float *o_partial, const float *lse,
                         int B, int Hq, int D, int S, cudaStream_t stream);
cudaError_t launch_append(const void *k_new, const void *v_new, int new_dtype, void *k_cache,
                          void *v_cache, int cache_dtype, float *k_scale, float *v_scale,
                          const int64_t *slot_mapping, int B, int Hkv, int D, int64_t num_blocks,
                          cudaStream_t stream);
cudaError_t launch_append_calibrated(const void *k_new, const void *v_new, int new_dtype, void *k_cache,
                                     void *v_cache, float *k_scale, float *v_scale, const int64_t *slot_mapping,
                                     int B, int Hkv, int D, int64_t num_blocks, cudaStream_t stream);
cudaError_t launch_copy(void *dst, const void *src, size_t bytes, int sm_count, cudaStream_t stream);
cudaError_t launch_copy_blocks(void *k_cache, void *v_cache, int cache_dtype, float *k_scale,
                               float *v_scale, const int32_t *pairs, int n_pairs, int Hkv, int D,
                               int64_t num_blocks, cudaStream_t stream);

}  // namespace pkv
