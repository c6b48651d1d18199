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
  return n;
}

}  // namespace pkv
