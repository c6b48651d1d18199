// decode_f16.cu — decode-attention kernel variants for f16 caches.
#include "decode.cuh"

namespace pkv {

int register_decode_f16(DecodeKernel *out) {
  int n = 0;
  out[n++] = decode_entry<DecodeCfg<F16, F16, 128, 8, true, kWarps, kBudget>>();
  out[n++] = decode_entry<DecodeCfg<F16, F16, 64, 8, true, kWarps, kBudget>>();
  out[n++] = decode_entry<DecodeCfg<F16, F16, 128, 2, false, kWarps, kBudget>>();
  out[n++] = decode_entry<DecodeCfg<F16, F16, 64, 2, false, kWarps, kBudget>>();
  out[n++] = decode_entry<DecodeCfg<F16, F16, 128, 1, false, kWarps, kBudget>>();
  out[n++] = decode_entry<DecodeCfg<F16, F16, 64, 1, false, kWarps, kBudget>>();
  // alternative pipeline shapes (PKV_DECODE_WARPS / PKV_DECODE_STAGES)
  out[n++] = decode_entry<DecodeCfg<F16, F16, 128, 8, true, 4, 16 * 1024>>();
  out[n++] = decode_entry<DecodeCfg<F16, F16, 128, 8, true, 6, 16 * 1024>>();
  out[n++] = decode_entry<DecodeCfg<F16, F16, 128, 8, true, 4, 24 * 1024>>();
  return n;
}

}  // namespace pkv
