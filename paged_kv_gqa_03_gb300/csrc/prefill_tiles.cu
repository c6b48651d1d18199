// prefill_tiles.cu — the tcgen05 prefill kernel with one CTA per work item
// (sequence, kv head, tile of 128 query rows): grid (row tiles, kv heads,
// sequences), the latest (heaviest) row tiles first, so the CTAs resident
// at one time share the K / V of few (sequence, kv head) pairs in L2.  Each
// CTA stages its Q tile, allocates tensor memory, streams its K / V tiles
// through the pipeline described in prefill_common.cuh and writes its rows.
// Chosen for long work items (a cached prefix of thousands of positions
// before the new tokens): there the per-tile loop of this kernel runs about
// 5-10% faster than the persistent kernel's, and the per-CTA start-up is
// small against the item.
#include "prefill.h"
#include "prefill_common.cuh"

namespace pkv {

// REP > 1 (a work item of at most 128 / REP query rows, e.g. a few new
// tokens of one GQA group): the tile holds REP replicas of the item's rows,
// and replica q takes the 16-position k-steps k with k mod REP = q of every
// K / V tile (its other P columns are written as zeros), so a softmax thread
// handles 64 / REP columns of a tile instead of 64; each replica keeps its
// own running max and sum, and the epilogue merges the REP partial rows
// (weights 2^(m_q - max m), through the then idle K ring).  The tensor work
// per tile is unchanged.
template <class Cfg, int REP>
__global__ void __launch_bounds__(Cfg::THREADS, 1)
    prefill_tile_kernel(const __grid_constant__ PrefillParams p, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t *sQ = smem;
  uint8_t *sK = sQ + Cfg::Q_BYTES;
  uint8_t *sV = sK + (size_t)Cfg::KSTAGES * Cfg::KV_BYTES;
  __shared__ __align__(8) uint64_t k_full[Cfg::KSTAGES], k_empty[Cfg::KSTAGES];
  __shared__ __align__(8) uint64_t v_full[Cfg::VSTAGES], v_empty[Cfg::VSTAGES];
  // per S buffer: S written, P written, P . V done.  (One P barrier per buffer:
  // the softmax may finish tile j + 1 before the MMA warp waits for tile j, but
  // it cannot finish tile j + SBUF before that.)
  __shared__ __align__(8) uint64_t s_full[Cfg::SBUF], p_full[Cfg::SBUF], pv_done[Cfg::SBUF], fin, xl;
  // row-max exchange per tile between the two warps holding the same rows (w, w + 4)
  __shared__ __align__(8) uint64_t xch[Cfg::SOFTMAX / 64][2];
  __shared__ __align__(8) uint64_t mrg[2];  // replica merge: (max, sum) written, partial O staged
  __shared__ __align__(8) uint64_t dead;
  static_assert(REP == 1 || REP == 2 || REP == 4, "replicas");
  constexpr int RW = Cfg::M / REP;  // query rows of one replica
  constexpr int KL = 4 / REP;       // k-steps of a replica in each half of a tile
  static_assert((REP - 1) * RW * Cfg::D * 4 <= Cfg::KSTAGES * Cfg::KV_BYTES, "replica staging");
  __shared__ float red[2][2][Cfg::M];  // partial row maxima [tile parity][half][row]
  __shared__ float red_l[2][Cfg::M];   // partial row sums [half][row]
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag, cta_flags, k_consumed, v_consumed, k_issued, v_issued;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile = p.max_tiles - 1 - (int)blockIdx.x;  // heaviest (latest) row tiles first
  const int h = blockIdx.y, b = blockIdx.z;
  const int qs = p.q_start ? __ldg(p.q_start + b) : b * p.uniform_q_len;
  const int n = p.q_start ? __ldg(p.q_start + b + 1) - qs : p.uniform_q_len;
  if (tid == 0 && tile == 0 && (n > p.max_q_len || n < 0) && p.status) atomicOr(p.status, PKV_FLAG_BAD_LEN);
  const int R = n * p.G;  // query rows of this kv head
  const int r0 = tile * Cfg::M;
  if (n <= 0 || r0 >= R) return;  // the whole CTA: no barrier or tensor memory touched yet

  const int ctx_raw = __ldg(p.context_lens + b);
  const int ctx = ctx_raw < 0 ? 0 : (ctx_raw > p.max_blocks * kBlock ? p.max_blocks * kBlock : ctx_raw);
  const int nblk = (ctx + kBlock - 1) / kBlock;
  const int i_lo = r0 / p.G, i_hi = min(R - 1, r0 + Cfg::M - 1) / p.G;
  const int lim_lo = ctx - n + i_lo + 1, lim_hi = ctx - n + i_hi + 1;  // exclusive causal ends
  const int first = p.window > 0 ? max(0, lim_lo - p.window) : 0;
  const int j_first = first / Cfg::N;
  const int T = lim_hi > 0 ? (lim_hi - 1) / Cfg::N - j_first + 1 : 0;  // K / V tiles to stream

  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < Cfg::KSTAGES; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
#pragma unroll
    for (int s = 0; s < Cfg::VSTAGES; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
#pragma unroll
    for (int s = 0; s < Cfg::SBUF; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&p_full[s], Cfg::SOFTMAX / 32);
      mbar_init(&pv_done[s], 1);
    }
#pragma unroll
    for (int pr = 0; pr < Cfg::SOFTMAX / 64; ++pr) {
      mbar_init(&xch[pr][0], 2);
      mbar_init(&xch[pr][1], 2);
    }
    mbar_init(&xl, Cfg::SOFTMAX / 32);
    mbar_init(&mrg[0], Cfg::SOFTMAX / 32);
    mbar_init(&mrg[1], Cfg::SOFTMAX / 32);
    mbar_init(&fin, 2);  // one commit from each issuing warp
    mbar_init(&dead, 1);  // failure-path test hook: nothing ever arrives on it
    fence_barrier_init();
    abort_flag = 0;
    cta_flags = ctx_raw != ctx ? PKV_FLAG_BAD_LEN : 0;
    k_consumed = v_consumed = k_issued = v_issued = 0;
  }
  if (warp == Cfg::ISSUER) tc::alloc(&tmem_base, Cfg::TMEM_COLS);
  if (warp == Cfg::PRODUCER && lane == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (tid < Cfg::SOFTMAX) {  // Q tile: thread (row, half) stages half of its row (zeros past R)
    const int row = tid & (Cfg::M - 1), half = tid / Cfg::M;
    const int r = r0 + row % RW;
    const int ii = r / p.G, g = r - ii * p.G;
    const uint4 *src = r < R ? reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(p.q) +
                                                             ((size_t)(qs + ii) * p.Hq + h * p.G + g) * Cfg::D)
                             : nullptr;
#pragma unroll
    for (int k = 0; k < Cfg::D / 16; ++k) {
      const int c = half * (Cfg::D / 16) + k;
      const uint4 v = src ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
      sts128(smem_u32(sQ + (c >> 3) * Cfg::PANEL_Q + row * 128 + (((c & 7) ^ (row & 7)) << 4)), v);
    }
    fence_proxy_async();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tbase = tmem_base;

  if (warp == Cfg::PRODUCER || warp == Cfg::V_PRODUCER) {
    // ---------------- TMA producers: K tiles (warp 8), V tiles (warp 10) ----------------
    // lane l fetches block (l % 8) of a tile, panel l / 8; block ids are
    // loaded three tiles ahead and first used when the tile's copies are
    // issued, so the loads' latency is hidden
    const int slot = lane & (Cfg::BLOCKS - 1), panel = lane / Cfg::BLOCKS;
    struct Pend {
      int id;
      bool none;  // past the context, or wholly before every row's window (such
                  // blocks may have been released): nothing to read
    };
    auto fetch = [&](int jj) -> Pend {
      const int lb = (j_first + jj) * Cfg::BLOCKS + slot;
      Pend f;
      f.none = jj >= T || lb >= nblk || (lb + 1) * kBlock <= first;
      f.id = f.none ? 0 : __ldg(p.block_table + (size_t)b * p.max_blocks + lb);
      return f;
    };
    int bad = 0;
    // the box row of a fetched block; the box past the tensor fills zeros
    auto row_of = [&](const Pend &f) -> int64_t {
      if (f.none) return p.num_blocks * p.Hkv;
      if (f.id >= 0 && (int64_t)f.id < p.num_blocks) return (int64_t)f.id * p.Hkv + h;
      bad = 1;
      return p.num_blocks * p.Hkv;
    };
    const bool vw = warp == Cfg::V_PRODUCER;
    Pend f0 = fetch(0), f1 = fetch(1), f2 = fetch(2);
    for (int j = 0; j < T; ++j) {
      const Pend f3 = fetch(j + 3);
      const int64_t trow = row_of(f0);
      if (!vw) {
        const int ks = j % Cfg::KSTAGES;
        if (j >= Cfg::KSTAGES &&
            !warp_wait(&k_empty[ks], (uint32_t)((j / Cfg::KSTAGES) - 1) & 1u, p.timeout_ns))
          break;
        if (__any_sync(kFull, *(volatile int *)&abort_flag)) break;
        if (lane == 0) mbar_arrive_expect_tx(&k_full[ks], Cfg::KV_BYTES);
        __syncwarp();
        if (lane < Cfg::LOADS)
          tma_load_2d(sK + (size_t)ks * Cfg::KV_BYTES + panel * Cfg::PANEL_KV + slot * 2048, &tmK, panel * 64,
                      (int)(trow * kBlock), &k_full[ks]);
        if (lane == 0) k_issued = j + 1;
      } else {
        const int vs = j % Cfg::VSTAGES;
        if (j >= Cfg::VSTAGES &&
            !warp_wait(&v_empty[vs], (uint32_t)((j / Cfg::VSTAGES) - 1) & 1u, p.timeout_ns))
          break;
        if (__any_sync(kFull, *(volatile int *)&abort_flag)) break;
        if (lane == 0) mbar_arrive_expect_tx(&v_full[vs], Cfg::KV_BYTES);
        __syncwarp();
        if (lane < Cfg::LOADS)
          tma_load_2d(sV + (size_t)vs * Cfg::KV_BYTES + panel * Cfg::PANEL_KV + slot * 2048, &tmV, panel * 64,
                      (int)(trow * kBlock), &v_full[vs]);
        if (lane == 0) v_issued = j + 1;
      }
      f0 = f1;
      f1 = f2;
      f2 = f3;
    }
    if (bad) atomicOr(&cta_flags, PKV_FLAG_BAD_BLOCK);
    if (__any_sync(kFull, (vw ? *(volatile int *)&v_issued : *(volatile int *)&k_issued) < T) && lane == 0 &&
        !*(volatile int *)&abort_flag) {
      atomicOr(&cta_flags, PKV_FLAG_TIMEOUT);
      abort_flag = 1;
    }
  } else if (warp == Cfg::ISSUER) {
    // ---------------- S issue (P . V has a warp of its own) ----------------
    const uint32_t q0 = smem_u32(sQ);
    bool ok = true;
    // S = Q . K^T of tile jj into S buffer jj % SBUF (free once P . V of tile
    // jj - SBUF, which read P from it, is done)
    auto issue_s = [&](int jj) -> bool {
      const int ks = jj % Cfg::KSTAGES, sb = jj % Cfg::SBUF;
      if (!warp_wait(&k_full[ks], (uint32_t)(jj / Cfg::KSTAGES) & 1u, p.timeout_ns)) return false;
      if (jj >= Cfg::SBUF &&
          !warp_wait(&pv_done[sb], (uint32_t)((jj / Cfg::SBUF) - 1) & 1u, p.timeout_ns))
        return false;
      if (lane == 0) k_consumed = jj + 1;
      tc::fence_after();
      if (lane == 0) {
        mma_s_tile<Cfg>(tbase + (uint32_t)(sb * Cfg::N), q0, smem_u32(sK + (size_t)ks * Cfg::KV_BYTES));
        tc::commit(&s_full[sb]);
        tc::commit(&k_empty[ks]);
      }
      __syncwarp();
      return true;
    };
    for (int j = 0; j < T && ok; ++j) {
      ok = issue_s(j);
      if (ok && __any_sync(kFull, *(volatile int *)&abort_flag)) ok = false;
    }
    if (!ok && lane == 0) {
      atomicOr(&cta_flags, PKV_FLAG_TIMEOUT);
      abort_flag = 1;
    }
  } else if (warp == Cfg::PV_ISSUER) {
    // ---------------- P . V issue ----------------
    bool ok = true;
    for (int j = 0; j < T; ++j) {
      const int vs = j % Cfg::VSTAGES, sb = j % Cfg::SBUF;
      ok = warp_wait(&v_full[vs], (uint32_t)(j / Cfg::VSTAGES) & 1u, p.timeout_ns);
      if (ok) ok = warp_wait(&p_full[sb], (uint32_t)(j / Cfg::SBUF) & 1u, p.timeout_ns);
      if (!ok) break;
      if (lane == 0) v_consumed = j + 1;
      uint8_t *vt = sV + (size_t)vs * Cfg::KV_BYTES;
      {  // stale cache rows past the context: weight 0, but 0 * NaN is NaN
        const int kv0 = (j_first + j) * Cfg::N;  // first position of the tile
        zero_v_rows<Cfg>(vt, ctx - kv0, min(nblk * kBlock - kv0, Cfg::N), lane);
      }
      __syncwarp();
      tc::fence_after();
      if (lane == 0) {
        mma_pv_tile<Cfg>(tbase + Cfg::COL_O, tbase + (uint32_t)(sb * Cfg::N), smem_u32(vt), j > 0);
        tc::commit(&pv_done[sb]);
        tc::commit(&v_empty[vs]);
      }
      __syncwarp();
      if (__any_sync(kFull, *(volatile int *)&abort_flag)) break;
    }
    if (!ok && lane == 0) {
      atomicOr(&cta_flags, PKV_FLAG_TIMEOUT);
      abort_flag = 1;
    }
  } else {
    // ---------------- softmax + epilogue: thread (row, half) ----------------
    constexpr int SC = Cfg::N / 2;  // S columns of a thread (its half of the row)
    constexpr int OC = Cfg::D / 2;  // O columns of a thread
    const int row = tid & (Cfg::M - 1), half = tid / Cfg::M;
    const int rr = row % RW, rep = row / RW;  // query row of the item, replica
    const int r = r0 + rr;
    const bool valid = r < R;
    const int lim = valid ? ctx - n + r / p.G + 1 : 0;  // visible positions [lo, lim)
    const int lo = (valid && p.window > 0) ? max(0, lim - p.window) : 0;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const float c = p.scale_log2;
    float m_run = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < T; ++j) {
      const int sb = j % Cfg::SBUF;
      // failure-path test hook: the first tile's wait is on a barrier
      // nothing completes, so it runs out and the CTA takes its abort path
      ok = (p.stall_ns != 0 && j == 0)
               ? warp_wait(&dead, 0, p.timeout_ns)
               : warp_wait(&s_full[sb], (uint32_t)(j / Cfg::SBUF) & 1u, p.timeout_ns);
      if (!ok) break;
      tc::fence_after();
      const uint32_t scol = tbase + lane_base + (uint32_t)(sb * Cfg::N + half * SC);
      // this thread's S values: all SC columns of its half (REP = 1), or the
      // KL k-steps rep, rep + REP, ... of its half (16 columns each)
      constexpr int NV = SC / REP;
      uint32_t s[NV];
      const int kvh = (j_first + j) * Cfg::N + half * SC;  // first position of this half
      if constexpr (REP == 1) {
#pragma unroll
        for (int q = 0; q < SC / 32; ++q)
          tc::ld32(scol + (uint32_t)(q * 32), *reinterpret_cast<uint32_t(*)[32]>(&s[q * 32]));
      } else {
#pragma unroll
        for (int t = 0; t < KL; ++t)
          tc::ld16(scol + (uint32_t)((rep + t * REP) * 16), *reinterpret_cast<uint32_t(*)[16]>(&s[t * 16]));
      }
      // position of value e: kvh + e (REP = 1), kvh + (rep + (e / 16) * REP) * 16 + e % 16
      auto pos_of = [&](int e) { return REP == 1 ? kvh + e : kvh + (rep + (e / 16) * REP) * 16 + (e & 15); };
      if (!(pos_of(0) >= lo && pos_of(NV - 1) < lim)) {  // a mask edge crosses these columns
#pragma unroll
        for (int e = 0; e < NV; ++e) {
          const int pos = pos_of(e);
          if (pos < lo || pos >= lim) s[e] = 0xff800000u;  // -inf
        }
      }
      float mx = -INFINITY;
#pragma unroll
      for (int e = 0; e < NV; e += 2) mx = fmax3(mx, __uint_as_float(s[e]), __uint_as_float(s[e + 1]));
      // the row max over both halves (double-buffered exchange, bounded wait)
      red[j & 1][half][row] = mx;
      __syncwarp();
      if (lane == 0) mbar_arrive(&xch[warp & 3][j & 1]);
      ok = warp_wait(&xch[warp & 3][j & 1], (uint32_t)(j >> 1) & 1u, p.timeout_ns);
      if (!ok) break;
      mx = fmaxf(mx, red[j & 1][half ^ 1][row]);
      const float m_new = fmaxf(m_run, mx * c);
      // warps w and w + 4 hold the same rows and the same m_new: same decision
      const bool rescale = __any_sync(kFull, m_new > m_run + 8.f);
      float alpha = 1.f;
      if (rescale) {
        alpha = m_new == -INFINITY ? 1.f : ex2(m_run - m_new);
        m_run = m_new;
      }
      const float mu = m_run == -INFINITY ? 0.f : m_run;
      const uint64_t cmu = f2_pack(c, c), nmu = f2_pack(-mu, -mu);
      uint64_t sum2 = f2_pack(0.f, 0.f);
      uint32_t w[NV / 2], wl[Cfg::BF ? NV / 2 : 1];
#pragma unroll
      for (int e = 0; e < NV / 2; ++e) {
        uint32_t lo_;
        p_pair<Cfg::BF>(s[2 * e], s[2 * e + 1], cmu, nmu, sum2, w[e], lo_);
        if constexpr (Cfg::BF) wl[e] = lo_;
      }
      const float2 sp = f2_unpack(sum2);
      const float sum = sp.x + sp.y;
      if (rescale && j > 0) {  // O must hold P . V of the previous tile before it is scaled
        ok = warp_wait(&pv_done[(j - 1) % Cfg::SBUF], (uint32_t)((j - 1) / Cfg::SBUF) & 1u, p.timeout_ns);
        if (!ok) break;
        tc::fence_after();
        scale_o<Cfg>(tbase + lane_base + Cfg::COL_O + (uint32_t)(half * OC), alpha);
      }
      l = l * alpha + sum;
      // P (bf16: high parts and residuals; f16: f16 pairs) over this thread's own (already read) S columns
      if constexpr (REP == 1) {
        tc::st32(scol, w);
        if constexpr (Cfg::BF) tc::st32(scol + 32, wl);
      } else {
        // 8 packed columns per k-step: this replica's k-steps, zeros in the others
#pragma unroll
        for (int t = 0; t < KL; ++t) {
          const uint32_t pc = scol + (uint32_t)((rep + t * REP) * 8);
          const uint32_t *v = &w[t * 8];
          tc::st8(pc, v[0], v[1], v[2], v[3], v[4], v[5], v[6], v[7]);
          if constexpr (Cfg::BF) {
            const uint32_t *u = &wl[t * 8];
            tc::st8(pc + 32, u[0], u[1], u[2], u[3], u[4], u[5], u[6], u[7]);
          }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (q % REP != rep) {
            tc::st8(scol + (uint32_t)(q * 8), 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u);
            if constexpr (Cfg::BF) tc::st8(scol + (uint32_t)(32 + q * 8), 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u);
          }
      }
      tc::wait_st();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[sb]);
    }
    if (ok && T > 0)
      ok = warp_wait(&pv_done[(T - 1) % Cfg::SBUF], (uint32_t)((T - 1) / Cfg::SBUF) & 1u, p.timeout_ns);
    if (ok) {  // the row sum over both halves
      red_l[half][row] = l;
      __syncwarp();
      if (lane == 0) mbar_arrive(&xl);
      ok = warp_wait(&xl, 0, p.timeout_ns);
    }
    if (!ok) {
      if (lane == 0) {
        atomicOr(&cta_flags, PKV_FLAG_TIMEOUT);
        abort_flag = 1;
      }
    } else {
      tc::fence_after();
      const float lt = l + red_l[half ^ 1][row];
      const int ii = r / p.G, g = r - ii * p.G;
      uint4 *dst = valid ? reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.out) +
                                                     ((size_t)(qs + ii) * p.Hq + h * p.G + g) * Cfg::D + half * OC)
                         : nullptr;
      if constexpr (REP == 1) {
        const float inv = lt > 0.f ? 1.f / lt : 0.f;  // a row that sees nothing gives 0
        uint32_t o[OC / 32][32];
#pragma unroll
        for (int q = 0; q < OC / 32; ++q) {
          if (T > 0) {
            tc::ld32(tbase + lane_base + Cfg::COL_O + (uint32_t)(half * OC + q * 32), o[q]);
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) o[q][e] = 0u;
          }
        }
        // staged in the K ring, idle now that every S has completed
        store_rows_staged<Cfg>(o, inv, dst, sK + (size_t)(warp * 2048), lane);
      } else if (T == 0) {  // no tile: every replica saw nothing
        if (dst && rep == 0) {
#pragma unroll
          for (int q = 0; q < OC / 8; ++q) dst[q] = make_uint4(0, 0, 0, 0);
        }
      } else {
        // merge the replicas of query row rr: weights 2^(m_q - M) / sum_q l_q 2^(m_q - M)
        float *mm = red[T & 1][0], *ml = red[T & 1][1];  // unused by the last tile's exchange
        if (half == 0) {
          mm[row] = m_run;
          ml[row] = lt;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&mrg[0]);
        ok = warp_wait(&mrg[0], 0, p.timeout_ns);
        if (ok) {
          float M = -INFINITY;
#pragma unroll
          for (int q = 0; q < REP; ++q) M = fmaxf(M, mm[q * RW + rr]);
          float L = 0.f;
#pragma unroll
          for (int q = 0; q < REP; ++q) {
            const float mq = mm[q * RW + rr];
            if (mq != -INFINITY) L += ml[q * RW + rr] * ex2(mq - M);
          }
          const float f = (m_run == -INFINITY || !(L > 0.f)) ? 0.f : ex2(m_run - M) / L;
          // replicas 1.. stage their weighted rows in the K ring (idle: every S
          // has completed), swizzled by 16-byte column groups
          float4 *stage = reinterpret_cast<float4 *>(sK);
          constexpr int C4 = Cfg::D / 4;  // float4 per staged row
          uint32_t o[OC / 32][32];
#pragma unroll
          for (int q = 0; q < OC / 32; ++q)
            tc::ld32(tbase + lane_base + Cfg::COL_O + (uint32_t)(half * OC + q * 32), o[q]);
          if (rep > 0) {
            float4 *srow = stage + (size_t)((rep - 1) * RW + rr) * C4;
#pragma unroll
            for (int q = 0; q < OC / 32; ++q)
#pragma unroll
              for (int v = 0; v < 8; ++v) {
                const int c4 = half * (OC / 4) + q * 8 + v;
                srow[c4 ^ (rr & 7)] = make_float4(__uint_as_float(o[q][4 * v]) * f, __uint_as_float(o[q][4 * v + 1]) * f,
                                                  __uint_as_float(o[q][4 * v + 2]) * f,
                                                  __uint_as_float(o[q][4 * v + 3]) * f);
              }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&mrg[1]);
          ok = warp_wait(&mrg[1], 0, p.timeout_ns);
          if (ok && rep == 0 && dst) {
#pragma unroll
            for (int q = 0; q < OC / 32; ++q)
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                float acc[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[e] = __uint_as_float(o[q][v * 8 + e]) * f;
#pragma unroll
                for (int k = 1; k < REP; ++k) {
                  const float4 *srow = stage + (size_t)((k - 1) * RW + rr) * C4;
                  const int c4 = half * (OC / 4) + q * 8 + 2 * v;
                  const float4 x0 = srow[c4 ^ (rr & 7)], x1 = srow[(c4 + 1) ^ (rr & 7)];
                  acc[0] += x0.x; acc[1] += x0.y; acc[2] += x0.z; acc[3] += x0.w;
                  acc[4] += x1.x; acc[5] += x1.y; acc[6] += x1.z; acc[7] += x1.w;
                }
                dst[q * 4 + v] = make_uint4(pack2<Cfg::BF>(acc[0], acc[1]), pack2<Cfg::BF>(acc[2], acc[3]),
                                            pack2<Cfg::BF>(acc[4], acc[5]), pack2<Cfg::BF>(acc[6], acc[7]));
              }
          }
        }
        if (!ok && lane == 0) {
          atomicOr(&cta_flags, PKV_FLAG_TIMEOUT);
          abort_flag = 1;
        }
      }
    }
  }

  // ---------------- drain, then free tensor memory ----------------
  tc::fence_before();
  __syncthreads();
  if (warp == Cfg::ISSUER || warp == Cfg::PV_ISSUER) {
    if (lane == 0) tc::commit(&fin);  // completes once every MMA either warp issued has
    __syncwarp();
    if (!mbar_wait_bounded(&fin, 0, p.timeout_ns) && lane == 0) atomicOr(&cta_flags, PKV_FLAG_TIMEOUT);
  } else if (warp == Cfg::PRODUCER && lane == 0) {  // copies issued but never consumed (abort only)
    for (int j = k_consumed; j < k_issued; ++j)
      mbar_wait_bounded(&k_full[j % Cfg::KSTAGES], (uint32_t)(j / Cfg::KSTAGES) & 1u, p.timeout_ns);
    for (int j = v_consumed; j < v_issued; ++j)
      mbar_wait_bounded(&v_full[j % Cfg::VSTAGES], (uint32_t)(j / Cfg::VSTAGES) & 1u, p.timeout_ns);
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == Cfg::ISSUER) tc::dealloc(tbase, Cfg::TMEM_COLS);
  if (tid == 0 && cta_flags && p.status) atomicOr(p.status, cta_flags);
}

template <class Cfg, int REP>
static cudaError_t launch_cfg(const PrefillParams &p, const CUtensorMap &tmK, const CUtensorMap &tmV,
                              cudaStream_t stream) {
  static int configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorNotSupported;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(prefill_tile_kernel<Cfg, REP>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg::SMEM);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  const dim3 grid((unsigned)p.max_tiles, (unsigned)p.Hkv, (unsigned)p.B);
  prefill_tile_kernel<Cfg, REP><<<grid, Cfg::THREADS, Cfg::SMEM, stream>>>(p, tmK, tmV);
  return cudaGetLastError();
}

// Replicas per tile: 4 when every item has at most 32 query rows
// (max_q_len * G <= 32), 2 when at most 64, else 1.
template <class Cfg>
static cudaError_t launch_rep(const PrefillParams &p, const CUtensorMap &tmK, const CUtensorMap &tmV,
                              cudaStream_t stream) {
  const int64_t rows = (int64_t)p.max_q_len * p.G;
  if (rows <= 32) return launch_cfg<Cfg, 4>(p, tmK, tmV, stream);
  if (rows <= 64) return launch_cfg<Cfg, 2>(p, tmK, tmV, stream);
  return launch_cfg<Cfg, 1>(p, tmK, tmV, stream);
}

cudaError_t launch_prefill_tiles(const PrefillParams &p, int cache_dtype, const CUtensorMap &tmK, const CUtensorMap &tmV,
                                 cudaStream_t stream) {
  if (p.max_tiles <= 0 || p.B <= 0) return cudaSuccess;
  if (cache_dtype == PKV_BF16) {
    if (p.D == 128) return launch_rep<PrefillCfg<BF16, 128>>(p, tmK, tmV, stream);
    if (p.D == 64) return launch_rep<PrefillCfg<BF16, 64>>(p, tmK, tmV, stream);
  } else if (cache_dtype == PKV_F16) {
    if (p.D == 128) return launch_rep<PrefillCfg<F16, 128>>(p, tmK, tmV, stream);
    if (p.D == 64) return launch_rep<PrefillCfg<F16, 64>>(p, tmK, tmV, stream);
  }
  return cudaErrorNotSupported;
}

}  // namespace pkv
