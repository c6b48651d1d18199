// decode_f16.cu — decode-attention kernel variants for f16 caches.
#include "decode.cuh"

namespace pkv {

int register_decode_f16(DecodeKernel *out) {
  int n = 0;
  // head dim 128: 6 warps x 16 KiB, 2 CTAs per SM (+0.9-1.1 % over 5 warps
  // on the fp16 MHA layer, whose short calls want more bytes in flight)
  out[n++] = decode_entry<DecodeCfg<F16, F16, 128, 8, true, 6, kBudget>>();
  out[n++] = decode_entry<DecodeCfg<F16, F16, 64, 8, true, kWarps, kBudget>>();
#ifdef PKV_SWEEP_SHAPES
  // for comparison runs and sweeps only, not in the product build: the
  // CUDA-core path on this cache type (PKV_PATH=simt) and alternative
  // pipeline shapes (warps per CTA, pipeline bytes per warp;
  // PKV_DECODE_WARPS / PKV_DECODE_STAGES)
  out[n++] = decode_entry<DecodeCfg<F16, F16, 128, 2, false, kWarps, kBudget>>();
  out[n++] = decode_entry<DecodeCfg<F16, F16, 64, 2, false, kWarps, kBudget>>();
  out[n++] = decode_entry<DecodeCfg<F16, F16, 128, 1, false, kWarps, kBudget>>();
  out[n++] = decode_entry<DecodeCfg<F16, F16, 64, 1, false, kWarps, kBudget>>();
  out[n++] = decode_entry<DecodeCfg<F16, F16, 128, 8, true, 4, 16 * 1024>>();
  out[n++] = decode_entry<DecodeCfg<F16, F16, 128, 8, true, 6, 16 * 1024>>();
  out[n++] = decode_entry<DecodeCfg<F16, F16, 128, 8, true, 4, 24 * 1024>>();
#endif
  return n;
}

}  // namespace pkv
