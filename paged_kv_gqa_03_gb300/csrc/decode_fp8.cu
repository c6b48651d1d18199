// decode_fp8.cu — decode-attention kernel variants for fp8-E4M3 caches
// (bf16 or f16 queries and outputs).
#include "decode.cuh"

namespace pkv {

// fp8 blocks carry half the bytes of bf16 ones for the same per-block work, so
// they want more warps in flight: 12 warps per SM with 16 KiB each.  With one
// block per stage (4 stages) 4 warps x 3 CTAs measured 5.91 TB/s on the
// long-context fp8 layer against 5.11 for 5 x 16 KiB x 2 CTAs, and it was
// issue-bound (half the bytes per instruction of the bf16 kernel); stages of
// two blocks (2 stages of 8 KiB) share the per-stage and per-softmax-update
// work between 32 tokens.  With two-block stages, 6 warps x 2 CTAs measured
// 0.5-0.6 % faster than 4 x 3 at head dim 128.
constexpr int kFp8Warps = 4;
constexpr int kFp8WideBudget = 24 * 1024;

int register_decode_fp8(DecodeKernel *out) {
  int n = 0;
  out[n++] = decode_entry<DecodeCfg<E4M3, BF16, 128, 8, true, 6, kBudget, 2>>();  // 6 x 16 KiB, 2 CTAs
  out[n++] = decode_entry<DecodeCfg<E4M3, BF16, 64, 8, true, kFp8Warps, kBudget, 2>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, F16, 128, 8, true, 6, kBudget, 2>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, F16, 64, 8, true, kFp8Warps, kBudget, 2>>();
  // 16-row units (kv heads with more than 8 query rows): twice the
  // accumulators and q fragments per warp, so two CTAs of 4 warps per SM
  // with 3 stages each
  out[n++] = decode_entry<DecodeCfg<E4M3, BF16, 128, 16, true, kFp8Warps, kFp8WideBudget, 2>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, BF16, 64, 16, true, kFp8Warps, kFp8WideBudget, 2>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, F16, 128, 16, true, kFp8Warps, kFp8WideBudget, 2>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, F16, 64, 16, true, kFp8Warps, kFp8WideBudget, 2>>();
#ifdef PKV_SWEEP_SHAPES
  // for comparison runs and sweeps only, not in the product build: the
  // CUDA-core path on this cache type (PKV_PATH=simt), one block per stage
  // (PKV_DECODE_STAGES=4) and alternative pipeline shapes (warps per CTA,
  // pipeline bytes per warp; PKV_DECODE_WARPS / PKV_DECODE_STAGES)
  out[n++] = decode_entry<DecodeCfg<E4M3, BF16, 128, 2, false, kWarps, kBudget>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, BF16, 64, 2, false, kWarps, kBudget>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, F16, 128, 2, false, kWarps, kBudget>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, F16, 64, 2, false, kWarps, kBudget>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, BF16, 128, 1, false, kWarps, kBudget>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, BF16, 64, 1, false, kWarps, kBudget>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, F16, 128, 1, false, kWarps, kBudget>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, F16, 64, 1, false, kWarps, kBudget>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, BF16, 128, 8, true, kFp8Warps, kBudget, 1>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, BF16, 128, 8, true, kFp8Warps, 24 * 1024, 2>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, BF16, 128, 8, true, 5, 16 * 1024, 2>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, BF16, 128, 8, true, 6, 16 * 1024, 2>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, BF16, 128, 8, true, 3, 24 * 1024, 2>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, BF16, 128, 16, true, 4, 16 * 1024, 2>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, BF16, 128, 16, true, 5, 16 * 1024, 2>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, BF16, 128, 16, true, 6, 16 * 1024, 2>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, BF16, 128, 16, true, 8, 16 * 1024, 2>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, BF16, 128, 16, true, 3, 24 * 1024, 2>>();
#endif
  return n;
}

}  // namespace pkv
