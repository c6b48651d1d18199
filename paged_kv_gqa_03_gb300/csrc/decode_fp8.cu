// decode_fp8.cu — decode-attention kernel variants for fp8-E4M3 caches
// (bf16 or f16 queries and outputs).
#include "decode.cuh"

namespace pkv {

// fp8 blocks carry half the bytes of bf16 ones for the same per-block work, so
// they want more warps in flight: 4 warps x 16 KiB (4 stages), 3 CTAs per SM
// measured 5.91 TB/s on the long-context fp8 layer against 5.11 for 5 x 16 KiB.
constexpr int kFp8Warps = 4;

int register_decode_fp8(DecodeKernel *out) {
  int n = 0;
  out[n++] = decode_entry<DecodeCfg<E4M3, BF16, 128, 8, true, kFp8Warps, kBudget>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, BF16, 64, 8, true, kFp8Warps, kBudget>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, F16, 128, 8, true, kFp8Warps, kBudget>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, F16, 64, 8, true, kFp8Warps, kBudget>>();
#ifdef PKV_SWEEP_SHAPES
  // for comparison runs and sweeps only, not in the product build: the
  // CUDA-core path on this cache type (PKV_PATH=simt) and alternative
  // pipeline shapes (warps per CTA, pipeline bytes per warp;
  // PKV_DECODE_WARPS / PKV_DECODE_STAGES)
  out[n++] = decode_entry<DecodeCfg<E4M3, BF16, 128, 2, false, kWarps, kBudget>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, BF16, 64, 2, false, kWarps, kBudget>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, F16, 128, 2, false, kWarps, kBudget>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, F16, 64, 2, false, kWarps, kBudget>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, BF16, 128, 1, false, kWarps, kBudget>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, BF16, 64, 1, false, kWarps, kBudget>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, F16, 128, 1, false, kWarps, kBudget>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, F16, 64, 1, false, kWarps, kBudget>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, BF16, 128, 8, true, 5, 16 * 1024>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, BF16, 128, 8, true, 6, 16 * 1024>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, BF16, 128, 8, true, 8, 12 * 1024>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, BF16, 128, 8, true, 4, 20 * 1024>>();
#endif
  return n;
}

}  // namespace pkv
