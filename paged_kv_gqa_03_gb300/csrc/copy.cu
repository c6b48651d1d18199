// copy.cu — pkv_copy: a byte copy performed by the SMs rather than a copy
// engine.  Either side may be pinned host memory (reachable from the GPU at
// the same address under unified addressing, over NVLink-C2C on Grace-based
// systems), which makes it the host<->device staging copy of a decode step:
// many CTAs issuing 16-byte loads move a step's ~1-2 MB of inputs faster than
// one small copy-engine transfer.
#include "common.cuh"
#include "internal.h"

namespace pkv {

__global__ void __launch_bounds__(256) copy16_kernel(uint4 *__restrict__ dst, const uint4 *__restrict__ src,
                                                     size_t n16) {
  grid_dep_wait();
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n16; i += 4 * stride) {  // four loads in flight per thread
    const uint4 a = src[i], b = src[i + stride], c = src[i + 2 * stride], d = src[i + 3 * stride];
    dst[i] = a;
    dst[i + stride] = b;
    dst[i + 2 * stride] = c;
    dst[i + 3 * stride] = d;
  }
  for (; i < n16; i += stride) dst[i] = src[i];
}

cudaError_t launch_copy(void *dst, const void *src, size_t bytes, int sm_count, cudaStream_t stream) {
  const size_t n16 = bytes / 16;
  if (n16 == 0) return cudaSuccess;
  // one 16-byte access per thread up to 16 CTAs per SM: host memory has a
  // long latency, so every load of a step-sized copy should be in flight at once
  size_t blocks = (n16 + 255) / 256;
  const size_t cap = (size_t)(sm_count > 0 ? sm_count : 148) * 16;
  if (blocks > cap) blocks = cap;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = stream != nullptr ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, copy16_kernel, static_cast<uint4 *>(dst), static_cast<const uint4 *>(src), n16);
}

}  // namespace pkv
