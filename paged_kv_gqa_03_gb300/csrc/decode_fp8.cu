// decode_fp8.cu — decode-attention kernel variants for fp8-E4M3 caches
// (bf16 or f16 queries and outputs).
#include "decode.cuh"

namespace pkv {

int register_decode_fp8(DecodeKernel *out) {
  int n = 0;
  out[n++] = decode_entry<DecodeCfg<E4M3, BF16, 128, 8, true, kWarps, kBudget>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, BF16, 64, 8, true, kWarps, kBudget>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, F16, 128, 8, true, kWarps, kBudget>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, F16, 64, 8, true, kWarps, kBudget>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, BF16, 128, 2, false, kWarps, kBudget>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, BF16, 64, 2, false, kWarps, kBudget>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, F16, 128, 2, false, kWarps, kBudget>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, F16, 64, 2, false, kWarps, kBudget>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, BF16, 128, 1, false, kWarps, kBudget>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, BF16, 64, 1, false, kWarps, kBudget>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, F16, 128, 1, false, kWarps, kBudget>>();
  out[n++] = decode_entry<DecodeCfg<E4M3, F16, 64, 1, false, kWarps, kBudget>>();
  return n;
}

}  // namespace pkv
