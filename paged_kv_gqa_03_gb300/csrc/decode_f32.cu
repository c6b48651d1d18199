// decode_f32.cu — decode-attention kernel variants for fp32 caches (CUDA cores).
#include "decode.cuh"

namespace pkv {

int register_decode_f32(DecodeKernel *out) {
  int n = 0;
  out[n++] = decode_entry<DecodeCfg<F32, F32, 128, 2, false, kWarps, kBudget>>();
  out[n++] = decode_entry<DecodeCfg<F32, F32, 64, 2, false, kWarps, kBudget>>();
  out[n++] = decode_entry<DecodeCfg<F32, F32, 128, 1, false, kWarps, kBudget>>();
  out[n++] = decode_entry<DecodeCfg<F32, F32, 64, 1, false, kWarps, kBudget>>();
  return n;
}

}  // namespace pkv
