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
// Plan kernel, for batches too large to plan inside the decode kernel:
// prefix[b] = sum_{b' < b} items_b' (ceil(ctx_b' / 16) blocks, less those
// before every row's sliding window); W = HU * prefix[B]; partition w starts at
// item floor(w * W / P), decoded into (b, hu, j).  One CTA; context
// lengths are clamped to [0, 16 * max_blocks] (flagged in plan_flags).
// ---------------------------------------------------------------------------
constexpr int kPlanSmemInts = 8192;  // prefix entries kept in shared memory (32 KiB)

__global__ void __launch_bounds__(1024) plan_kernel(const DecodeParams p) {
  grid_dep_launch();  // the decode kernel may start its prologue now
  __shared__ int32_t warp_tot[32];
  __shared__ int32_t carry, s_flags;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nw = blockDim.x >> 5;
  if (tid == 0) {
    carry = 0;
    s_flags = 0;
  }
  __syncthreads();
  int flags = 0;
  for (int base = 0; base < p.B; base += blockDim.x) {
    const int b = base + tid;
    int n = 0;
    if (b < p.B) {
      const int ctx = p.context_lens[b];
      if (ctx < 0 || ctx > p.max_blocks * kBlock) flags |= PKV_FLAG_BAD_LEN;
      n = seq_items(p, clamped_len(p, ctx));
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
  if (flags) atomicOr(&s_flags, flags);
  __syncthreads();
  if (tid == 0) {
    p.prefix[p.B] = total_blocks;
    p.hdr->plan_flags = s_flags;
  }
  __syncthreads();  // prefix[B] is read below by other threads
  const int64_t W = (int64_t)p.HU * total_blocks;
  const int64_t Pe = active_partitions(p, W);
  if (tid == 0) {
    p.hdr->P = p.P;
    p.hdr->W = (int32_t)W;
    p.hdr->B = p.B;
    p.hdr->HU = p.HU;
  }
  // the binary searches read the prefix from shared memory when it fits
  extern __shared__ int32_t s_prefix[];
  const bool in_smem = p.B + 1 <= kPlanSmemInts;
  if (in_smem) {
    for (int b = tid; b <= p.B; b += blockDim.x) s_prefix[b] = p.prefix[b];
    __syncthreads();
  }
  const int32_t *pre = in_smem ? s_prefix : p.prefix;
  for (int w = tid; w <= p.P; w += blockDim.x) {
    const int64_t s = w < Pe ? W * w / Pe : W;
    int4 r;
    if (s >= W) {
      r = make_int4((int)W, p.B, 0, 0);
    } else {
      int lo = 0, hi = p.B - 1;  // largest b with HU * prefix[b] <= s
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((int64_t)p.HU * pre[mid] <= s)
          lo = mid;
        else
          hi = mid - 1;
      }
      const int n = pre[lo + 1] - pre[lo];
      const int64_t rr = s - (int64_t)p.HU * pre[lo];
      const int j0 = first_block(p, clamped_len(p, p.context_lens[lo]));
      r = make_int4((int)s, lo, (int)(rr / n), j0 + (int)(rr % n));
    }
    p.starts[w] = r;
  }
}

cudaError_t launch_plan(const DecodeParams &p, cudaStream_t stream) {
  const size_t smem = p.B + 1 <= kPlanSmemInts ? sizeof(int32_t) * (size_t)(p.B + 1) : 0;
  plan_kernel<<<1, 1024, smem, stream>>>(p);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Merge kernel for the partials of units that a partition boundary cut (a8),
// launched behind the decode kernel with programmatic dependent launch.  One
// CTA per unit; a unit processed whole by one warp was already written.  Partition w covers
// items [floor(w W / P), floor((w+1) W / P)) — the plan kernel's rule,
// recomputed.  Segments are taken in chunks whose partial indices are staged
// in shared memory; each thread keeps an online max / sum for its row and
// accumulates 4 head-dim elements of every partial with one 16-byte load,
// eight partials' LSE and output loads in flight at a time (a long context
// cut over many warps — the 32K fp8 layer has ~14 partials per unit — would
// otherwise pay one L2 latency per partial in sequence).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void store4_out(int dtype, void *p, size_t i, float4 v) {
  if (dtype == PKV_F32) {
    *reinterpret_cast<float4 *>(static_cast<float *>(p) + i) = v;
  } else if (dtype == PKV_F16) {
    const uint32_t lo = pack_f16x2(v.x, v.y), hi = pack_f16x2(v.z, v.w);
    *reinterpret_cast<uint2 *>(static_cast<__half *>(p) + i) = make_uint2(lo, hi);
  } else {
    const uint32_t lo = pack_bf16x2(v.x, v.y), hi = pack_bf16x2(v.z, v.w);
    *reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(p) + i) = make_uint2(lo, hi);
  }
}

__global__ void __launch_bounds__(512) splitk_merge_kernel(const DecodeParams p) {
  constexpr int kSegChunk = 32;
  constexpr int kBatch = 8;  // partials whose loads are in flight together
  __shared__ int32_t s_base[kSegChunk];  // partial index of each segment of a chunk (-1: none)
  grid_dep_wait();
  if (blockIdx.x == 0 && threadIdx.x < 32) {  // publish the call's status bits
    int f = p.inline_plan ? 0 : p.hdr->plan_flags;
    for (int c = threadIdx.x; c < p.n_ctas; c += 32) f |= p.cta_flags[c];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) f |= __shfl_xor_sync(kFull, f, off);
    if (threadIdx.x == 0) {
      p.hdr->status = f;
      p.hdr->P = p.P;
      p.hdr->W = p.HU * p.prefix[p.B];
      p.hdr->B = p.B;
      p.hdr->HU = p.HU;
    }
  }
  const int u = blockIdx.x;
  const int b = u / p.HU, hu = u % p.HU;
  const int h = hu / p.NC, r0 = (hu % p.NC) * p.GC;
  const int gc = min(p.GC, p.R - r0);
  const int D = p.D;
  const int pb = p.prefix[b];
  const int n = p.prefix[b + 1] - pb;
  const int nvec = gc * D / 4;  // float4s of the unit's rows: <= blockDim.x
  // output offset of row r0 + g of this unit ([B][q_len][Hq][D])
  auto out_row = [&](int g) {
    const int r = r0 + g, i = r / p.G;
    return (((size_t)b * p.q_len + i) * p.Hq + h * p.G + (r - i * p.G)) * (size_t)D;
  };
  const int v = threadIdx.x;
  const int g = (4 * v) / D, d = (4 * v) % D;
  if (n == 0) {  // nothing to attend: the output is zero
    if (v < nvec) store4_out(p.out_dtype, p.out, out_row(g) + d, make_float4(0.f, 0.f, 0.f, 0.f));
    return;
  }
  const int64_t W = (int64_t)p.HU * p.prefix[p.B];
  const int64_t Pe = active_partitions(p, W);
  const int64_t a = (int64_t)p.HU * pb + (int64_t)hu * n, e = a + n;
  const int wf = (int)(((a + 1) * Pe - 1) / W);
  const int wl = (int)((e * Pe - 1) / W);
  if (wf == wl) return;

  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float M = -INFINITY, den = 0.f;
  for (int cs = wf; cs <= wl; cs += kSegChunk) {
    const int ns = min(kSegChunk, wl - cs + 1);
    __syncthreads();  // the previous chunk's segment table has been read
    for (int sgi = threadIdx.x; sgi < ns; sgi += blockDim.x) {
      const int w = cs + sgi;
      const int64_t sw = W * w / Pe, ew = W * (w + 1) / Pe;
      const bool valid = (a > sw ? a : sw) < (e < ew ? e : ew);
      const int slot = sw >= a ? 0 : 1;
      s_base[sgi] = valid ? (int32_t)(((int64_t)w * 2 + slot) * p.GC) : -1;  // [worker][slot][GC rows]
    }
    __syncthreads();
    if (v >= nvec) continue;
    // a batch of partials: their lse and output loads are issued together,
    // so the L2 latencies overlap; the batch then joins the running merge
    for (int s0 = 0; s0 < ns; s0 += kBatch) {
      float4 o[kBatch];
      float l[kBatch];
#pragma unroll
      for (int t = 0; t < kBatch; ++t) {
        const int base = s0 + t < ns ? s_base[s0 + t] : -1;
        l[t] = base >= 0 ? p.part_lse[base + g] : -INFINITY;
        o[t] = base >= 0 ? *reinterpret_cast<const float4 *>(p.part_o + ((size_t)base + g) * D + d)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      float cm = -INFINITY;
#pragma unroll
      for (int t = 0; t < kBatch; ++t) cm = fmaxf(cm, l[t]);
      if (cm == -INFINITY) continue;  // no partial of the batch saw a position of this row
      const float mn = fmaxf(M, cm);
      const float rescale = exp2f(M - mn);
      acc.x *= rescale; acc.y *= rescale; acc.z *= rescale; acc.w *= rescale;
      den *= rescale;
#pragma unroll
      for (int t = 0; t < kBatch; ++t) {
        const bool on = l[t] != -INFINITY;  // empty partials weigh 0 (and are not read)
        const float wt = on ? exp2f(l[t] - mn) : 0.f;
        acc.x = fmaf(wt, on ? o[t].x : 0.f, acc.x);
        acc.y = fmaf(wt, on ? o[t].y : 0.f, acc.y);
        acc.z = fmaf(wt, on ? o[t].z : 0.f, acc.z);
        acc.w = fmaf(wt, on ? o[t].w : 0.f, acc.w);
        den += wt;
      }
      M = mn;
    }
  }
  if (v < nvec) {
    const float inv = den > 0.f ? 1.f / den : 0.f;  // no visible position: 0
    store4_out(p.out_dtype, p.out, out_row(g) + d, make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv));
  }
}

cudaError_t launch_splitk_merge(const DecodeParams &p, cudaStream_t stream, bool pdl) {
  const int units = p.B * p.HU;
  if (units == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  // one float4 of a unit's rows per thread (D <= 128): as many threads as the
  // widest unit has float4s (an MHA unit has one row, 32 float4s at D = 128;
  // a 16-row fp8 unit 512)
  const int rows = p.GC < p.R ? p.GC : p.R;
  const int threads = (rows * p.D / 4 + 31) / 32 * 32;
  cfg.gridDim = dim3(units);
  cfg.blockDim = dim3(threads < 32 ? 32 : threads);
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
