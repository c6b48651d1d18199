/*
 * pagedkv.h — C ABI of libpagedkv.so: single-token decode attention over a
 * paged (block_size 16) KV cache with GQA/MQA head groups, for sm_103a.
 *
 * What the library computes, per decode step:
 *
 *   out[b, hq, :] = softmax_t( scale * q[b, hq, :] . K_b,h[t, :] ) . V_b,h[t, :]
 *   for t < context_lens[b], h = hq / (Hq / Hkv)
 *
 * This is scaled dot-product attention for one new query row
 * ("苦猿的大模型日记 Day45", PART 02: Attention(Q,K,V) = softmax(QK^T/sqrt(d))V;
 * "LLM推理优化实战：从KV-Cache到Continuous Batching", §1.1 attention_step),
 * evaluated against a KV cache that lives in fixed-size physical blocks reached
 * through a per-sequence block table ("LLM推理优化实战", §2.2 PageAttention,
 * BLOCK_SIZE = 16; "大模型推理加速核心KV Cache 复用机制与内存布局优化", §三
 * BlockTable), with groups of query heads sharing one KV head ("大模型推理加速
 * ——KV Cache篇", §6.2 MHA/GQA/MQA).
 *
 * Conventions shared by every entry point
 *  - Block size is fixed at PKV_BLOCK_SIZE = 16 tokens.
 *  - Cache layout: k_cache and v_cache are separate dense arrays
 *    [num_blocks][Hkv][16][D] (D fastest).  A (block, kv-head) tile of 16 tokens
 *    is therefore one contiguous 16*D-element run.
 *  - q, out: [B][Hq][D]; k_new, v_new: [B][Hkv][D]; all dense row-major.
 *  - Query head hq reads kv head hq / (Hq/Hkv) (consecutive groups).
 *  - FP8 caches (PKV_FP8_E4M3, OCP "e4m3fn": max 448, no infinities) carry one
 *    fp32 scale per (block, kv-head), separately for K and V:
 *    k_scale, v_scale: [num_blocks][Hkv]; element value = decode(byte) * scale.
 *  - context_lens[b] is the attended length INCLUDING the token appended this
 *    step; the appended token sits at position context_lens[b]-1.
 *  - Every pointer argument that names a tensor is a DEVICE pointer unless the
 *    entry point says otherwise.  The caller owns all memory; the library never
 *    allocates device memory and keeps no per-call state outside `workspace`.
 *  - Calls are asynchronous on `stream` (NULL = the legacy default stream) and
 *    never synchronise the host, except where a function says so.
 *  - Every function returns a pkv_status_t (0 = success, negative = error).
 *    Arguments are validated before anything is launched: a call that returns
 *    PKV_EINVAL / PKV_EUNSUPPORTED / PKV_EWORKSPACE has touched no memory.
 *    PKV_ECUDA means a CUDA runtime call failed; pkv_last_cuda_error() returns
 *    its cudaError_t.  Nothing is thrown across this boundary.
 *  - Tensor pointers handed to the TMA engine (k_cache, v_cache, q, out and
 *    workspace) must be 16-byte aligned.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream; NULL selects the legacy default stream. */
typedef struct CUstream_st *pkv_stream_t;

#define PKV_BLOCK_SIZE 16

typedef enum {
  PKV_F32 = 0,
  PKV_F16 = 1,
  PKV_BF16 = 2,
  PKV_FP8_E4M3 = 3
} pkv_dtype_t;

typedef enum {
  PKV_OK = 0,
  PKV_EINVAL = -1,        /* a null pointer, a negative size, Hq % Hkv != 0, ... */
  PKV_EUNSUPPORTED = -2,  /* a valid but unimplemented shape or dtype combination */
  PKV_EWORKSPACE = -3,    /* workspace missing, misaligned or too small */
  PKV_ECUDA = -4,         /* a CUDA runtime call failed (see pkv_last_cuda_error) */
  PKV_ETIMEOUT = -5,      /* a bounded in-kernel wait gave up (see paged_decode_status) */
  PKV_EOOM = -6,          /* block manager: no free physical block */
  PKV_ERANGE = -7,        /* a block id, slot or length outside its table */
  PKV_ENOTFOUND = -8      /* block manager: unknown sequence id */
} pkv_status_t;

/* Status bits that kernels record in the workspace header (paged_decode_status). */
#define PKV_FLAG_TIMEOUT 1   /* a pipeline wait exceeded its time limit */
#define PKV_FLAG_BAD_LEN 2   /* context_lens[b] < 0 or > 16 * max_blocks_per_seq (clamped) */
#define PKV_FLAG_BAD_BLOCK 4 /* a block-table entry outside [0, num_blocks) (read as zeros) */
#define PKV_FLAG_RANGE 8     /* reserved: a value outside the range a kernel can represent (no kernel raises it) */

/* ------------------------------------------------------------------------ */
/* Step a3 — KV append through a slot mapping.                              */
/* ------------------------------------------------------------------------ */
/*
 * Writes the new token's K/V rows into the paged cache:
 *   k_cache[slot / 16][h][slot % 16][:] = k_new[b][h][:]   (same for V)
 * with slot = slot_mapping[b] (int64, device).  slot < 0 means "padding, skip";
 * a slot whose block is >= num_blocks is skipped as well.
 * The write is the KV-cache update of incremental decoding ("大模型推理加速——KV
 * Cache篇", §3.1 Attention.forward step 2; "苦猿的大模型日记 Day45", PART 02,
 * new_k/new_v appended to the cache), addressed through the block table
 * ("LLM推理优化实战", §2.2, logical block = num_tokens // BLOCK_SIZE).
 *
 * Types: for PKV_F32/F16/BF16 caches new_dtype must equal cache_dtype and the
 * copy is bit-exact.  For a PKV_FP8_E4M3 cache, new_dtype is F32, F16 or BF16
 * and each element is stored as e4m3(round-to-nearest-even, saturating to
 * +-448)(x / scale) with the division done in fp32.  The scale is the block's
 * existing k_scale/v_scale entry, except when slot % 16 == 0 (the token opens a
 * fresh block): then scale = max_d |x_d| / 448 (1.0 if that is 0) is computed
 * from the token and written to k_scale/v_scale first.  k_scale and v_scale are
 * required (non-NULL) exactly when cache_dtype is PKV_FP8_E4M3.
 * Slots must be distinct within one call.  Several tokens of one sequence may
 * be appended in one call (q_len new tokens, see paged_decode_attention_multi)
 * when they are consecutive entries of slot_mapping in position order (what
 * pkv_bm_append_slots returns for an id repeated consecutively): a token of a
 * block opened earlier in the same call then uses the opener's scale, exactly
 * as if the tokens had been appended one call at a time.  With an FP8 cache,
 * other orders that put a block's opener and a later token of it in one call
 * are not supported.
 */
int paged_kv_append(const void *k_new, const void *v_new, int new_dtype,
                    void *k_cache, void *v_cache, int cache_dtype,
                    float *k_scale, float *v_scale,
                    const int64_t *slot_mapping,
                    int B, int Hkv, int D, int64_t num_blocks,
                    pkv_stream_t stream);

/*
 * paged_kv_append with calibrated FP8 block scales (the FP8 calibration that
 * "苦猿的大模型日记 Day45" PART 02 and "大模型推理加速核心KV Cache 复用机制与内存
 * 布局优化" §四 say decides an FP8 cache's quality).  Same arguments.  For an
 * FP8 cache a block's scale is the smallest power of two p with
 * max|x| <= 448 p over the tokens written to the block so far: a token at
 * offset 0 sets it; a later token whose own p is larger raises the scale and
 * first re-quantises the block's earlier bytes to
 *   e4m3_rne_sat( fp32( decode(q) * p_old ) / p_new ),
 * an exact exponent shift for values in the e4m3 normal range; each token is
 * stored as e4m3_rne_sat(x / p) (fp32 division).  No stored value saturates.
 * Tokens are applied in slot_mapping order; several tokens of one block in one
 * call must be consecutive entries in position order (pkv_bm_append_slots
 * order).  Blocks written with the plain rule may be continued with this one
 * (their scale is then raised to a power of two only if a token outgrows it).
 * Other cache types: exactly paged_kv_append.
 */
int paged_kv_append_calibrated(const void *k_new, const void *v_new, int new_dtype,
                               void *k_cache, void *v_cache, int cache_dtype,
                               float *k_scale, float *v_scale,
                               const int64_t *slot_mapping, int B, int Hkv, int D,
                               int64_t num_blocks, pkv_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Steps a4–a8 — paged gather, scores, online softmax, PV, split-KV merge.  */
/* ------------------------------------------------------------------------ */
/*
 * Size in bytes of the workspace paged_decode_attention needs for these shapes
 * on the CURRENT device; written to *bytes_out.  num_splits has the meaning it
 * has for paged_decode_attention.
 */
int paged_decode_workspace_bytes(int B, int Hq, int Hkv, int D,
                                 int cache_dtype, int q_dtype, int num_splits,
                                 size_t *bytes_out);

/*
 * Decode attention for one query token per sequence.
 *
 *   out        [B][Hq][D], dtype = q_dtype (fp32 results rounded to nearest even);
 *              device memory, or pinned host memory (cudaHostAlloc / torch
 *              pin_memory, addressed by the GPU under unified addressing):
 *              the kernels then write the rows over the host link, which
 *              spares a device-to-host copy of the output (any entry point
 *              that writes `out`: the multi-query and prefill calls too)
 *   q          [B][Hq][D]; q_dtype: F32 with an F32 cache, else F16/BF16;
 *              must equal cache_dtype for F16/BF16 caches.
 *   k_cache, v_cache  [num_blocks][Hkv][16][D] of cache_dtype
 *   k_scale, v_scale  [num_blocks][Hkv] fp32, FP8 caches only (else NULL)
 *   block_table       [B][max_blocks_per_seq] int32 physical block ids
 *   context_lens      [B] int32 attended lengths (0 gives out = 0)
 *   scale             the softmax temperature, normally 1/sqrt(D)
 *   D                 64 or 128
 *
 * Work decomposition (GB300 design, not taken from the pages): the
 * concatenation of every (sequence, kv-head) block list is cut into
 * `num_splits` contiguous, equally long partitions, one per warp (a kv head
 * with more query rows than a unit holds — 8, or 16 on FP8 caches — has one
 * block list per unit of rows); a warp
 * streams its blocks through a TMA pipeline and keeps an fp32 online softmax
 * (running max m, running sum l, rescaled accumulator — "LLM推理优化实战", §3.2
 * flash_attention online softmax).  Partitions that cover only part of a
 * sequence leave (o, lse) partials that a merge kernel combines with the
 * log-sum-exp rule (flash-decoding split-KV, named in "苦猿的大模型日记 Day45"
 * PART 03; the inter-block merge of "大模型推理加速核心KV Cache 复用机制与内存
 * 布局优化" §四).  num_splits = 0 picks one partition per resident warp of the
 * current GPU; any positive value is allowed and gives the same result up to
 * fp32 rounding.
 *
 * workspace: device memory of at least paged_decode_workspace_bytes(...) bytes,
 * 256-byte aligned, owned by the caller, reused across calls; concurrent calls
 * must use distinct workspaces.  It needs no initialisation.
 */
int paged_decode_attention(void *out, const void *q, int q_dtype,
                           const void *k_cache, const void *v_cache, int cache_dtype,
                           const float *k_scale, const float *v_scale,
                           const int32_t *block_table, int max_blocks_per_seq,
                           const int32_t *context_lens,
                           int B, int Hq, int Hkv, int D, int64_t num_blocks,
                           float scale, int num_splits,
                           void *workspace, size_t workspace_bytes,
                           pkv_stream_t stream);

/*
 * Decode attention for q_len new query tokens per sequence (the verify step
 * of speculative decoding, "LLM推理优化实战" §4, or a chunked decode step).
 * The q_len tokens are the newest q_len positions of each sequence and are
 * already in the cache (appended with paged_kv_append, slots in order), so
 * context_lens[b] counts them.  New token i (0-based) attends positions
 * 0 .. ctx_b - q_len + i: the causal mask tril(ones(q_len, ctx), diagonal =
 * ctx - q_len) of the naive_attention in "苦猿的大模型日记 Day45" PART 04.
 * A row that sees no position (ctx_b < q_len - i) gives out = 0.
 *
 * Sliding window (window W > 0; 0 = none): each row sees only the W most
 * recent positions up to its own, [lim - W, lim) with lim = ctx_b - q_len + i
 * + 1 — the fixed visible history of "苦猿的大模型日记 Day45" PART 02 (sliding
 * window / KV eviction).  Only blocks that hold a position some row of the
 * sequence sees are read (the first is the block of ctx_b - q_len + 1 - W), so
 * entries of block_table before it may be -1 (see pkv_bm_release_window).
 *
 *   q, out     [B][q_len][Hq][D] (q_len = 1 is paged_decode_attention)
 *   q_len      1 .. PKV_MAX_Q_LEN
 *   window     0 (no window) or W >= 1 (W >= 2^30 acts as no window)
 *   max_blocks_per_seq  at most 2^26 (PKV_EUNSUPPORTED above), for every
 *              decode entry point
 * Everything else, including the workspace rule, is as for
 * paged_decode_attention; the workspace size comes from
 * paged_decode_multi_workspace_bytes (which covers every kernel below).
 * Kernels, all meeting the same error bound; with q_len >= 2, an F16 or BF16
 * cache, num_splits = 0 and scale > 0:
 *  - R = q_len * G <= 32 query rows per kv head, D = 128, B <= 2048: a
 *    tensor-core kernel with the cache positions on the MMA's M side (S^T =
 *    K . Q^T, O^T = V^T . P^T), one CTA per SM over equal shares of all
 *    (sequence, kv head) K/V tiles (any batch shape fills the GPU) and a
 *    merge of the (sequence, kv head) items cut between CTAs; each K/V byte is
 *    read once for all R rows;
 *  - R <= 64 the same, unless the tensor-core prefill kernel's grid (below)
 *    fills the SMs;
 *  - otherwise, with at least one (sequence, kv head, 128-row tile) per SM,
 *    a tensor-core prefill kernel (chosen as in paged_prefill_attention),
 *    which also reads each (sequence, kv head)'s K/V once for all its rows;
 *  - otherwise (FP8 and F32 caches, a fixed split count, small grids) each
 *    kv head's rows are served in units by the decode kernel (K/V read once
 *    per unit, re-reads mostly from L2) with the split-KV merge: units of 8
 *    rows, or of 16 rows on an FP8 cache with more than 8 rows per kv head
 *    (each E4M3 element widened to f16 once per 16 rows).
 * pkv_set_route(PKV_ROUTE_MULTI_QUERY, PKV_MQ_TRANSPOSED | PKV_MQ_PREFILL |
 * PKV_MQ_UNITS) forces the first, second or last route where it applies
 * (measurement and tests).  Forced, the first route also takes an FP8 cache
 * with up to 32 rows and D = 128: its producer warps copy the E4M3 tiles
 * and its softmax warps widen each to f16 in shared memory (exact), the
 * block scales multiplying the scores and folded into the weights (slower
 * than the 16-row units on GB300, hence not automatic).
 */
#define PKV_MAX_Q_LEN 64
int paged_decode_multi_workspace_bytes(int B, int q_len, int Hq, int Hkv, int D,
                                       int cache_dtype, int q_dtype, int num_splits,
                                       size_t *bytes_out);
int paged_decode_attention_multi(void *out, const void *q, int q_dtype,
                                 const void *k_cache, const void *v_cache, int cache_dtype,
                                 const float *k_scale, const float *v_scale,
                                 const int32_t *block_table, int max_blocks_per_seq,
                                 const int32_t *context_lens,
                                 int B, int q_len, int window, int Hq, int Hkv, int D,
                                 int64_t num_blocks, float scale, int num_splits,
                                 void *workspace, size_t workspace_bytes,
                                 pkv_stream_t stream);

/*
 * Paged prefill attention on the tensor cores (tcgen05): sequence b's
 * n_b = q_start[b+1] - q_start[b] new tokens — its prompt, or a chunk of it
 * after a cached prefix — attend causally over its paged cache.  The tokens
 * are already appended (paged_kv_append, slots in order) and are the n_b
 * newest of ctx_b = context_lens[b] positions: new token i (position
 * ctx_b - n_b + i) attends positions 0 .. ctx_b - n_b + i, or only the
 * `window` most recent of them when window > 0.  This is FlashAttention's
 * tiled computation ("LLM推理优化实战" §3.2 flash_attention: row blocks of Q,
 * blocks of K / V, online softmax) with the causal mask of "苦猿的大模型日记
 * Day45" PART 04; a row that sees nothing gives 0.
 *
 *   q, out       [total][Hq][D], total = q_start[B]; rows of sequence b start
 *                at q_start[b] (int32 [B+1], device, non-decreasing, q_start[0] = 0)
 *   q_dtype      must equal cache_dtype, which is PKV_F16 or PKV_BF16
 *                (PKV_EUNSUPPORTED otherwise; FP8 caches use the decode path)
 *   max_q_len    >= every n_b (host value; sizes the grid); a larger n_b sets
 *                PKV_FLAG_BAD_LEN and rows past max_q_len are not written
 *   scale        > 0 (PKV_EINVAL otherwise)
 *   window       0 (none) or W >= 1
 *   status       device int32 or NULL: zeroed by the call, then the OR of
 *                PKV_FLAG_* bits (bad block id, bad length, in-kernel timeout)
 *   D            64 or 128; B <= 65535
 * Other arguments as for paged_decode_attention.  Asynchronous on `stream`;
 * needs no workspace.
 *
 * P . V takes V exactly as stored.  For a bf16 cache the attention weights
 * enter it as a bf16 high part plus its bf16 residual (two MMAs per 16
 * positions, ~16 significant bits; bf16 alone would give 8), for an f16 cache
 * as f16: every V value of either type is used as it is, over its type's
 * whole range.
 *
 * Two kernels run the same tile pipeline: one CTA per (128-row tile, kv
 * head, sequence), chosen when max_blocks_per_seq * 16 - max_q_len >= 2048
 * (the table admits a long cached prefix, so the items are long; 1024 when
 * max_q_len * Hq / Hkv <= 64, where it runs row replicas), and one
 * persistent CTA per SM walking those items otherwise (prompts: many short
 * items of unequal length).  pkv_set_route(PKV_ROUTE_PREFILL,
 * PKV_PREFILL_PER_ITEM | PKV_PREFILL_PERSISTENT) overrides the choice;
 * results agree within the tolerance either way.
 */
int paged_prefill_attention(void *out, const void *q, int q_dtype,
                            const void *k_cache, const void *v_cache, int cache_dtype,
                            const int32_t *block_table, int max_blocks_per_seq,
                            const int32_t *context_lens, const int32_t *q_start,
                            int B, int max_q_len, int Hq, int Hkv, int D, int64_t num_blocks,
                            float scale, int window, int32_t *status, pkv_stream_t stream);

/*
 * paged_decode_attention for callers that cannot allocate device memory.
 * The pages have no counterpart to this entry point; it exists for callers of
 * this library.  Some of them cannot hand over a workspace: a plain C host
 * program without a device allocator of its own, a plugin or custom operator
 * whose host framework owns all device memory and offers no scratch, or a
 * serving loop that must not call cudaMalloc once running (it can synchronise
 * the device and can fail under a fixed memory budget).
 *
 * Same operation, arguments, layouts and results as paged_decode_attention,
 * without `workspace` / `workspace_bytes`: the scratch comes from one array of
 * PKV_STATIC_SCRATCH_BYTES bytes that the library keeps in device memory on
 * every GPU that loads it, until the process exits.
 *  - Limit: with num_splits > 0, a shape whose
 *    paged_decode_workspace_bytes() exceeds PKV_STATIC_SCRATCH_BYTES is
 *    rejected with PKV_EWORKSPACE before anything runs.  With num_splits = 0
 *    the library takes its usual partition count (one per resident warp) when
 *    that fits (16 MiB holds D = 128 with 8-row units and ~2000 partitions),
 *    else the largest count that fits (FP8 caches with more than 8 query rows
 *    per kv head keep 16-row partials, 16 KiB a partition at D = 128); only a
 *    shape that does not fit with one partition is rejected.
 *  - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *  - Set-up: every call looks up the array's device address in the current
 *    device's context (cudaGetSymbolAddress, a host-side lookup that
 *    allocates nothing), so the address stays right after a cudaDeviceReset.
 *    The first call on a device also loads the library's device code there;
 *    make that first call before any stream capture.
 *  - Sharing: every call on a device uses the same array, which keeps the last
 *    call's contents.  Nothing in it has to start at zero (each call writes
 *    what it later reads), so it is never cleared.  Calls that overlap on the
 *    GPU (several streams or host threads) race on the array: serialise them.
 *  - Status: paged_decode_static_status() reads the status bits the last
 *    call on the current device recorded in the array (timeouts, bad block
 *    ids, clamped lengths).  After a call whose status is not PKV_OK the
 *    output may hold partial results of an earlier call: check it before
 *    using the output when the inputs are not trusted.
 */
#define PKV_STATIC_SCRATCH_BYTES (16u << 20)
int paged_decode_attention_static(void *out, const void *q, int q_dtype,
                                  const void *k_cache, const void *v_cache, int cache_dtype,
                                  const float *k_scale, const float *v_scale,
                                  const int32_t *block_table, int max_blocks_per_seq,
                                  const int32_t *context_lens,
                                  int B, int Hq, int Hkv, int D, int64_t num_blocks,
                                  float scale, int num_splits,
                                  pkv_stream_t stream);

/*
 * paged_decode_status() for paged_decode_attention_static: synchronises
 * `stream` and reads the status bits of the last static call on the current
 * device (the array every such call shares).  Same returns as
 * paged_decode_status.  No counterpart on the pages.
 */
int paged_decode_static_status(pkv_stream_t stream, int *flags_out);

/*
 * Synchronises `stream` and reads the status bits (PKV_FLAG_*) that the last
 * paged_decode_attention on `workspace` recorded.  Returns PKV_ETIMEOUT if
 * PKV_FLAG_TIMEOUT is set, PKV_ERANGE if a range flag is set, else PKV_OK;
 * *flags_out (may be NULL) receives the raw bits.  This is the one call that
 * blocks the host.
 */
int paged_decode_status(const void *workspace, size_t workspace_bytes,
                        pkv_stream_t stream, int *flags_out);

/*
 * Log-sum-exp merge of S partial attention results per (b, hq) row:
 *   M = max_s lse[b][hq][s];  w_s = exp(lse[b][hq][s] - M)
 *   out[b][hq][:] = sum_s w_s * o_partial[b][hq][s][:] / sum_s w_s
 * o_partial [B][Hq][S][D] fp32 (each partial already normalised by its own
 * softmax sum), lse [B][Hq][S] fp32 natural-log log-sum-exp of the partial's
 * scaled scores; lse = -inf marks an empty partial, and a row whose partials
 * are all empty gives out = 0.  out dtype is out_dtype (F32, F16 or BF16).
 * The rule follows from the online-softmax rescaling identity ("LLM推理优化实
 * 战", §3.2: O·exp(m_old - m_new) + ..., l·exp(m_old - m_new) + ...).
 */
int paged_decode_merge(void *out, int out_dtype,
                       const float *o_partial, const float *lse,
                       int B, int Hq, int D, int S,
                       pkv_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Step a2 — copy-on-write block copy.                                      */
/* ------------------------------------------------------------------------ */
/*
 * For each pair i: cache[dst_i] = cache[src_i] for all kv heads of both K and
 * V (and the fp8 scales when cache_dtype is PKV_FP8_E4M3), where
 * src_dst_pairs = {src_0, dst_0, src_1, dst_1, ...} (int32, device).  This is
 * the copy that copy-on-write performs before a shared block is written
 * ("LLM推理优化实战", §2.2 Copy-on-Write; "大模型推理加速——KV Cache篇", §6.1).
 * Pairs with an id outside [0, num_blocks) are skipped.  Destinations must be
 * distinct and must not appear as sources in the same call.
 */
int paged_kv_copy_blocks(void *k_cache, void *v_cache, int cache_dtype,
                         float *k_scale, float *v_scale,
                         const int32_t *src_dst_pairs, int n_pairs,
                         int Hkv, int D, int64_t num_blocks,
                         pkv_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Route overrides (measurement and tests).                                 */
/* ------------------------------------------------------------------------ */
/*
 * The library picks its kernels by a fixed rule of each call's shapes (see
 * paged_decode_attention_multi and paged_prefill_attention); nothing in it
 * reads the environment.  pkv_set_route replaces that rule for one decision,
 * process-wide, until the decision is set back to PKV_ROUTE_AUTO, so that
 * tests can run each kernel on the same inputs and measurements can compare
 * them.  A forced route applies only where the chosen kernel supports the
 * call (otherwise the automatic rule decides).  Each call reads the setting
 * once; change it only while no call is being issued on another host thread.
 *   which = PKV_ROUTE_MULTI_QUERY (q_len >= 2 decode):
 *           PKV_ROUTE_AUTO, PKV_MQ_TRANSPOSED (the transposed tensor-core
 *           kernel), PKV_MQ_PREFILL (the 128-row prefill kernel), PKV_MQ_UNITS
 *           (the decode kernel's 8- or 16-row units with the split-KV merge)
 *   which = PKV_ROUTE_PREFILL (the prefill kernel's schedule):
 *           PKV_ROUTE_AUTO, PKV_PREFILL_PERSISTENT, PKV_PREFILL_PER_ITEM
 * Returns PKV_EINVAL for an unknown `which` or `choice`; pkv_get_route
 * returns the current setting (or PKV_EINVAL).
 */
#define PKV_ROUTE_MULTI_QUERY 0
#define PKV_ROUTE_PREFILL 1
#define PKV_ROUTE_AUTO 0
#define PKV_MQ_TRANSPOSED 1
#define PKV_MQ_PREFILL 2
#define PKV_MQ_UNITS 3
#define PKV_PREFILL_PERSISTENT 1
#define PKV_PREFILL_PER_ITEM 2
int pkv_set_route(int which, int choice);
int pkv_get_route(int which);

/* ------------------------------------------------------------------------ */
/* Failure-path test hook.                                                  */
/* ------------------------------------------------------------------------ */
/*
 * Makes the next call that launches the given kernel family take its timeout
 * path, so that tests can check that path without a fault or a hang.  In that
 * call every bounded in-kernel wait is limited to limit_ns (normally 4 s), and
 *  - PKV_STALL_DECODE (the decode kernel: paged_decode_attention, and the
 *    unit route of paged_decode_attention_multi): the worker holding the
 *    first work item replaces its first pipeline wait by a wait on a barrier
 *    that nothing completes;
 *  - PKV_STALL_PREFILL (either prefill kernel, from paged_prefill_attention or
 *    the multi-query route): the softmax warps of every CTA with work replace
 *    their first wait for S by such a wait.
 * That wait gives up after limit_ns; the CTA records PKV_FLAG_TIMEOUT, lets
 * the copies and tensor-core operations it has in flight complete (waiting
 * within the same limit), frees its tensor memory and exits; its outputs are
 * left incomplete.  The call's status (paged_decode_status, or the prefill
 * status word) reports the timeout, and the workspace is fit for the next
 * call.  One-shot: the next call that launches the family consumes the
 * request; limit_ns = 0 cancels it.  limit_ns must lie in [1e6, 1e10]
 * (1 ms .. 10 s), else PKV_EINVAL.  For tests of the failure path only.
 */
#define PKV_STALL_DECODE 0
#define PKV_STALL_PREFILL 1
int pkv_test_stall_next(int which, uint64_t limit_ns);

/* ------------------------------------------------------------------------ */
/* Staging copy.                                                            */
/* ------------------------------------------------------------------------ */
/*
 * dst[0:bytes] = src[0:bytes], performed by the SMs (a kernel on `stream`)
 * rather than a copy engine.  Either pointer may be pinned host memory
 * (cudaHostAlloc / torch pin_memory), which the GPU addresses directly under
 * unified addressing — over NVLink-C2C on Grace-based systems — so this is the
 * host<->device staging copy of a decode step (its inputs in, its output
 * out): for the ~1-2 MB a step moves, many CTAs issuing 16-byte accesses beat
 * one copy-engine transfer.  Both pointers and `bytes` must be 16-byte
 * aligned; the ranges must not overlap.
 */
int pkv_copy(void *dst, const void *src, size_t bytes, pkv_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Step a1 — host block manager: allocate / fork / free / slot mapping.     */
/* ------------------------------------------------------------------------ */
/*
 * A host-side (CPU) physical-block allocator with per-sequence block tables and
 * reference counts, after the BlockTable of "大模型推理加速核心KV Cache 复用机制
 * 与内存布局优化" §三: the free list starts as [0, 1, ..., num_blocks-1] and
 * hands out blocks from its END (LIFO); allocate() takes ceil(n/16) blocks or
 * fails without change; fork() shares the parent's blocks (refcount + 1);
 * free() decrements and returns blocks whose count reaches 0 to the end of the
 * free list, in table order.  All pointers in this section are HOST pointers.
 * A manager is not thread-safe; use one per thread or lock around it.
 */
typedef struct pkv_block_manager pkv_block_manager;

/* Creates a manager over num_blocks physical blocks; NULL on failure. */
pkv_block_manager *pkv_bm_create(int64_t num_blocks);
void pkv_bm_destroy(pkv_block_manager *bm);

/* allocate(seq, num_tokens): fresh table of ceil(num_tokens/16) blocks
 * (refcount 1).  PKV_EOOM (no change) if the free list is too short,
 * PKV_EINVAL if seq already exists or num_tokens < 0. */
int pkv_bm_allocate(pkv_block_manager *bm, int64_t seq, int64_t num_tokens);

/* Adopts an explicit block list for a new sequence holding num_tokens tokens
 * (refcount + 1 per block; blocks leave the free list, which keeps the order
 * of the remaining entries).  Used to mirror tables built elsewhere, and to
 * share one prefix among many sequences.  nblocks must equal
 * ceil(num_tokens/16); PKV_ERANGE for an id outside [0, num_blocks). */
int pkv_bm_adopt(pkv_block_manager *bm, int64_t seq, const int32_t *blocks,
                 int nblocks, int64_t num_tokens);

/* fork(parent, child): the child gets a copy of the parent's table and token
 * count; every block's refcount + 1.  PKV_ENOTFOUND / PKV_EINVAL on bad ids. */
int pkv_bm_fork(pkv_block_manager *bm, int64_t parent, int64_t child);

/* free(seq): refcount - 1 per block, blocks at 0 go back to the free list. */
int pkv_bm_free(pkv_block_manager *bm, int64_t seq);

/* Sliding window (KV eviction, "苦猿的大模型日记 Day45" PART 02: a fixed cache
 * bound in exchange for visible history): with window W >= 1 the sequence's
 * next token (position tokens(seq)) and every later one see only positions
 * >= tokens(seq) + 1 - W, so every block whose 16 positions all lie below that
 * is released: refcount - 1 (back to the end of the free list at 0, in table
 * order) and its table entry becomes -1 (exported as -1; fork and free skip
 * it).  The table keeps its length, so logical block j stays entry j.  Call it
 * before a step's pkv_bm_append_slots with the window that step's
 * paged_decode_attention_multi uses; *released_out (may be NULL) receives the
 * number of entries released.  PKV_EINVAL for W < 1, PKV_ENOTFOUND for an
 * unknown id. */
int pkv_bm_release_window(pkv_block_manager *bm, int64_t seq, int64_t window,
                          int64_t *released_out);

/*
 * Reserves the slot of one new token for each of the n sequences seqs[i]:
 *   pos = tokens(seq); if pos % 16 == 0 a fresh block is appended to the table;
 *   else if the block holding pos is shared (refcount > 1) it is replaced by a
 *   fresh block and the pair (old, new) is reported for a copy (copy-on-write);
 *   slot_out[i] = table[pos / 16] * 16 + pos % 16;  tokens(seq) = pos + 1.
 * cow_pairs_out (capacity 2*n int32) receives {src, dst, ...}; *n_cow_out the
 * number of pairs.  On PKV_EOOM / PKV_ENOTFOUND every sequence is left as it
 * was before the call.
 */
int pkv_bm_append_slots(pkv_block_manager *bm, const int64_t *seqs, int n,
                        int64_t *slot_out, int32_t *cow_pairs_out, int *n_cow_out);

/* Exports the block tables of n sequences as a dense [n][max_blocks] int32
 * array (unused entries = -1) and their token counts as int32 context
 * lengths.  PKV_ERANGE if a table is longer than max_blocks. */
int pkv_bm_export(const pkv_block_manager *bm, const int64_t *seqs, int n,
                  int32_t *table_out, int max_blocks, int32_t *context_lens_out);

int64_t pkv_bm_num_free(const pkv_block_manager *bm);
/* Refcount of a physical block (-1 for an id out of range). */
int pkv_bm_refcount(const pkv_block_manager *bm, int64_t block);
/* Token count of a sequence (-1 if unknown). */
int64_t pkv_bm_num_tokens(const pkv_block_manager *bm, int64_t seq);

/* ------------------------------------------------------------------------ */
/* Diagnostics.                                                             */
/* ------------------------------------------------------------------------ */
const char *pkv_status_string(int status);
/* cudaError_t of the last PKV_ECUDA returned on the calling thread (0 if none). */
int pkv_last_cuda_error(void);
/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int pkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
