// mq_decode.h — host side of the transposed tensor-core multi-query decode
// (mq_decode.cu): q_len new tokens per sequence, q_len * G <= 64 query rows
// per kv head (32 for fp8 caches), head dim 128, 16-bit or fp8 caches.
#pragma once

#include "internal.h"

namespace pkv {

constexpr int kMqRows = 64;         // most query rows (q_len * G) per kv head
constexpr int kMqMaxBatch = 2048;   // sequences: each CTA keeps their tile prefix in shared memory
constexpr int kMqHeadDim = 128;
constexpr int kMqRowsFp8 = 32;      // fp8 caches: most query rows (shared memory also holds the raw tiles)

struct MqParams {
  void *out;                    // [B][q_len][Hq][D], the query's 16-bit type
  const void *q;                // [B][q_len][Hq][D]
  const float *k_scale;         // fp8 caches: [num_blocks][Hkv] block scales (else null)
  const float *v_scale;
  const int32_t *block_table;   // [B][max_blocks]
  const int32_t *context_lens;  // [B], the appended tokens included
  int32_t *status;              // PKV_FLAG_* bits of the call (written by the merge kernel)
  int32_t *cta_flags;           // [grid] workspace: each CTA's PKV_FLAG_* bits
  int32_t *prefix;              // [B + 1] workspace: K / V tiles before sequence b, over all kv heads
  float *part_o;                // [grid][2][kMqRows][D] normalised partial outputs of split items
  float *part_lse;              // [grid][2][kMqRows], log2 domain
  int64_t num_blocks;
  int B, q_len, Hq, Hkv, G, R, max_blocks, window;
  float scale_log2;             // softmax scale * log2(e), > 0
  uint64_t timeout_ns;
};

// Workspace of one call: the WsHeader (status) at offset 0, then the tile
// prefix and the partial outputs of `grid` CTAs.
struct MqWsLayout {
  size_t prefix, cta_flags, part_o, part_lse, total;
};
MqWsLayout mq_ws_layout(int B, int grid);

// Launches the decode kernel (grid CTAs, one per SM) and, for grid > 1, the
// merge of items split between CTAs.  cudaErrorNotSupported for a shape the
// kernel is not built for.
cudaError_t launch_mq_decode(const MqParams &p, int cache_dtype, int q_dtype, const CUtensorMap &tmK,
                             const CUtensorMap &tmV, int grid, cudaStream_t stream);

}  // namespace pkv
