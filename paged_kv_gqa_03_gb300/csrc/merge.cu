// merge.cu — the plan kernel that cuts the decode work into partitions, the
// merge of partition partials (step a8), and the exported generic merge.
//
// Merge rule: partial p of a query row carries its normalised output o_p and
// lse_p = log-sum-exp of its scaled scores; with M = max_p lse_p,
//   out = sum_p exp(lse_p - M) o_p / sum_p exp(lse_p - M),
// which follows from the online-softmax rescaling ("LLM推理优化实战" §3.2:
// O and l are rescaled by exp(m_old - m_new) when the running max grows) and
// is the inter-block merge that paged kernels need ("大模型推理加速核心KV Cache
// 复用机制与内存布局优化" §四).
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace pkv {

// ---------------------------------------------------------------------------
// Plan: prefix[b] = sum_{b' < b} ceil(ctx_b' / 16); W = HU * prefix[B];
// partition w starts at item floor(w * W / P), decoded into (b, hu, j).
// One CTA; context lengths are clamped to [0, 16 * max_blocks] (flagged).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) plan_kernel(const DecodeParams p) {
  grid_dep_launch();  // the decode kernel may start its prologue now
  __shared__ int32_t warp_tot[32];
  __shared__ int32_t carry;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nw = blockDim.x >> 5;
  if (tid == 0) carry = 0;
  __syncthreads();
  int flags = 0;
  for (int base = 0; base < p.B; base += blockDim.x) {
    const int b = base + tid;
    int n = 0;
    if (b < p.B) {
      int ctx = p.context_lens[b];
      if (ctx < 0 || ctx > p.max_blocks * kBlock) flags |= PKV_FLAG_BAD_LEN;
      ctx = ctx < 0 ? 0 : (ctx > p.max_blocks * kBlock ? p.max_blocks * kBlock : ctx);
      n = (ctx + kBlock - 1) / kBlock;
    }
    int x = n;  // inclusive scan within the warp
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(kFull, x, off);
      if (lane >= off) x += y;
    }
    if (lane == 31) warp_tot[wid] = x;
    __syncthreads();
    if (wid == 0) {
      const int v = lane < nw ? warp_tot[lane] : 0;
      int incl = v;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(kFull, incl, off);
        if (lane >= off) incl += y;
      }
      if (lane < nw) warp_tot[lane] = incl - v;  // exclusive warp offsets
    }
    __syncthreads();
    const int excl = carry + warp_tot[wid] + x - n;
    if (b < p.B) p.prefix[b] = excl;
    __syncthreads();
    if (tid == blockDim.x - 1) carry = excl + n;
    __syncthreads();
  }
  const int total_blocks = carry;
  if (tid == 0) {
    p.prefix[p.B] = total_blocks;
    p.hdr->status = 0;
  }
  __syncthreads();
  if (flags) atomicOr(&p.hdr->status, flags);
  const int64_t W = (int64_t)p.HU * total_blocks;
  if (tid == 0) {
    p.hdr->P = p.P;
    p.hdr->W = (int32_t)W;
    p.hdr->B = p.B;
    p.hdr->HU = p.HU;
  }
  for (int w = tid; w <= p.P; w += blockDim.x) {
    const int64_t s = W * w / p.P;
    int4 r;
    if (s >= W) {
      r = make_int4((int)W, p.B, 0, 0);
    } else {
      int lo = 0, hi = p.B - 1;  // largest b with HU * prefix[b] <= s
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((int64_t)p.HU * p.prefix[mid] <= s)
          lo = mid;
        else
          hi = mid - 1;
      }
      const int n = p.prefix[lo + 1] - p.prefix[lo];
      const int64_t rr = s - (int64_t)p.HU * p.prefix[lo];
      r = make_int4((int)s, lo, (int)(rr / n), (int)(rr % n));
    }
    p.starts[w] = r;
  }
}

cudaError_t launch_plan(const DecodeParams &p, cudaStream_t stream) {
  plan_kernel<<<1, 1024, 0, stream>>>(p);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Merge of the partials of units that a partition boundary cut.  One CTA per
// unit; a unit processed whole by one warp was already written.  Units of
// empty sequences are written as zeros here.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128) splitk_merge_kernel(const DecodeParams p) {
  grid_dep_wait();
  const int u = blockIdx.x;
  const int b = u / p.HU, hu = u % p.HU;
  const int h = hu / p.NC, c = hu % p.NC;
  const int head0 = h * p.G + c * p.GC;
  const int gc = min(p.GC, p.G - c * p.GC);
  const int pb = p.prefix[b];
  const int n = p.prefix[b + 1] - pb;
  if (n == 0) {
    for (int idx = threadIdx.x; idx < gc * p.D; idx += blockDim.x)
      store_out(p.out_dtype, p.out, ((size_t)b * p.Hq + head0) * p.D + idx, 0.f);
    return;
  }
  const int64_t W = (int64_t)p.HU * p.prefix[p.B];
  const int64_t a = (int64_t)p.HU * pb + (int64_t)hu * n, e = a + n;
  const int wf = (int)(((a + 1) * p.P - 1) / W);
  const int wl = (int)((e * p.P - 1) / W);
  if (wf == wl) return;
  for (int idx = threadIdx.x; idx < gc * p.D; idx += blockDim.x) {
    const int g = idx / p.D, d = idx % p.D;
    float M = -INFINITY;
    for (int w = wf; w <= wl; ++w) {
      const int64_t sw = p.starts[w].x, ew = p.starts[w + 1].x;
      if ((a > sw ? a : sw) < (e < ew ? e : ew)) {
        const int slot = sw >= a ? 0 : 1;
        M = fmaxf(M, p.part_lse[((size_t)w * 2 + slot) * kChunkMax + g]);
      }
    }
    float num = 0.f, den = 0.f;
    for (int w = wf; w <= wl; ++w) {
      const int64_t sw = p.starts[w].x, ew = p.starts[w + 1].x;
      if ((a > sw ? a : sw) < (e < ew ? e : ew)) {
        const int slot = sw >= a ? 0 : 1;
        const size_t base = ((size_t)w * 2 + slot) * kChunkMax + g;
        const float wt = exp2f(p.part_lse[base] - M);
        num = fmaf(wt, p.part_o[base * p.D + d], num);
        den += wt;
      }
    }
    store_out(p.out_dtype, p.out, ((size_t)b * p.Hq + head0 + g) * p.D + d, num / den);
  }
}

cudaError_t launch_splitk_merge(const DecodeParams &p, cudaStream_t stream, bool pdl) {
  const int units = p.B * p.HU;
  if (units == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(units);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, splitk_merge_kernel, p);
}

// ---------------------------------------------------------------------------
// Exported generic merge: rows of S partials, natural-log lse, -inf = empty.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128) merge_kernel(void *out, int out_dtype, const float *o_partial,
                                                    const float *lse, int D, int S) {
  const size_t row = blockIdx.x;
  const float *l = lse + row * S;
  float M = -INFINITY;
  for (int s = 0; s < S; ++s) M = fmaxf(M, l[s]);
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float num = 0.f, den = 0.f;
    if (M != -INFINITY) {
      for (int s = 0; s < S; ++s) {
        if (l[s] == -INFINITY) continue;
        const float wt = expf(l[s] - M);
        num = fmaf(wt, o_partial[(row * S + s) * D + d], num);
        den += wt;
      }
    }
    store_out(out_dtype, out, row * D + d, den > 0.f ? num / den : 0.f);
  }
}

cudaError_t launch_merge(void *out, int out_dtype, const float *o_partial, const float *lse, int B, int Hq,
                         int D, int S, cudaStream_t stream) {
  const size_t rows = (size_t)B * Hq;
  if (rows == 0) return cudaSuccess;
  merge_kernel<<<(unsigned)rows, 128, 0, stream>>>(out, out_dtype, o_partial, lse, D, S);
  return cudaGetLastError();
}

}  // namespace pkv
