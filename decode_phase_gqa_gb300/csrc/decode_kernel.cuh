// Split-KV flash-decoding kernel over a paged KV cache (second launch of a step).
//
// Work decomposition.  Every (sequence b, KV head j, query-head group) is a
// "stream" of ceil((L_b + 1) / 16) units of 16 cached tokens.  The streams are
// laid end to end and the flattened unit list is cut into n_active equal,
// contiguous shares, one per CTA, so every CTA reads the same number of bytes
// whatever the length mix (the skewed long-context batches included).  A
// stream that lies inside one share is finished by its CTA; one cut across
// shares leaves a partial softmax state (m, l, acc) per share and the last CTA
// to arrive (atomic counter, no waiting) merges them by log-sum-exp.
//
// Inside a CTA each of the 4 warps owns every 4th unit of the share and runs
// its own ring of bulk (TMA) copies: one elected lane issues
// cp.async.bulk of the contiguous [16][d] K and V blocks (plus their int8
// scales) into shared memory, completing on a per-stage mbarrier.  A unit's
// K/V block is read from shared memory once and reused by all query heads of
// the group (GQA sharing: "Qwen3-8B inference engine from scratch in
// C++/CUDA", section 4.4.2 "GQA grouped decode").  Scores are
// dot(q_h, k_t) * scale ("LLM inference from smollm3.go", section
// "Self-attention"), kept in log2 units (the query arrives pre-multiplied by
// scale * log2 e); softmax is the online form in fp32 with warp shuffles; the
// weighted value sum accumulates in fp32 registers.
//
// Lane layout for a unit: 8 consecutive head-dim elements per lane (16 bytes of
// bf16 or 8 bytes of int8), LPR = d/8 lanes per token row, RPP = 32/LPR rows
// per pass.  Each lane keeps the partial dot products of all its rows and
// heads and the warp reduces them with a transposing butterfly (every level
// halves the values a lane keeps), so a unit costs 30 shuffles instead of one
// full reduction per (row, head).
#pragma once

#include <map>
#include <mutex>
#include <set>
#include <utility>

#include "kvattn_internal.cuh"

namespace kvattn {

template <int D, int GS, bool INT8>
struct DecodeCfg {
  static constexpr int kESize = INT8 ? 1 : 2;
  static constexpr int kLPR = D / 8;
  static constexpr int kRPP = 32 / kLPR;
  static constexpr int kNPass = kUnitRows / kRPP;
  static constexpr int kNV = kNPass * GS;
  static constexpr int kNVL = kNV >= kLPR ? kNV / kLPR : 1;
  static constexpr int kHPL = (GS + 1) / 2;  // softmax heads per lane
  static constexpr int kTile = kUnitRows * D * kESize;
  static constexpr int kScaleBytes = INT8 ? kUnitRows * 4 : 0;
  static constexpr int kStage = 2 * kTile + 2 * kScaleBytes;
  static constexpr int kSW = (72 * 1024) / (kDecodeWarps * kStage) > 8
                                 ? 8
                                 : (72 * 1024) / (kDecodeWarps * kStage);
  static constexpr int kStagesBytes = kDecodeWarps * kSW * kStage;
  static constexpr int kBarBytes = kDecodeWarps * kSW * 8;
  static constexpr int kScBytes = kDecodeWarps * kUnitRows * GS * 4;
  static constexpr int kMergeBytes = kDecodeWarps * GS * (D + 2) * 4;
  static constexpr int kMiscBytes = 64;
  static constexpr int kFixedSmem = kStagesBytes + kBarBytes + kScBytes + kMergeBytes + kMiscBytes;
  static_assert(kStage % 128 == 0, "stage must keep 128-byte alignment");
  static_assert(kSW >= 2, "need at least double buffering");
};

// transposing butterfly: N values per lane reduced over the lanes whose index
// differs in bits M, M/2, ..., 1; afterwards value i of lane l holds the sum of
// original index i + (l % (2M)) * N / (2M)   (or l % (2M) * N / (2M) when N < 2M)
template <int N, int M>
struct TransposeReduce {
  __device__ __forceinline__ static void run(float *v, int lane) {
    if constexpr (M == 0) {
      return;
    } else if constexpr (N == 1) {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], M);
      TransposeReduce<1, M / 2>::run(v, lane);
    } else {
      const bool upper = (lane & M) != 0;
#pragma unroll
      for (int i = 0; i < N / 2; ++i) {
        const float send = upper ? v[i] : v[i + N / 2];
        const float keep = upper ? v[i + N / 2] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, M);
      }
      TransposeReduce<N / 2, M / 2>::run(v, lane);
    }
  }
};

template <bool INT8>
__device__ __forceinline__ void load_row8(const uint8_t *src, float (&f)[8]) {
  if constexpr (INT8) {
    const uint2 r = *reinterpret_cast<const uint2 *>(src);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      f[k] = static_cast<float>(static_cast<int8_t>(r.x >> (8 * k)));
      f[4 + k] = static_cast<float>(static_cast<int8_t>(r.y >> (8 * k)));
    }
  } else {
    const uint4 r = *reinterpret_cast<const uint4 *>(src);
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      f[2 * k] = __uint_as_float(w[k] << 16);
      f[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
    }
  }
}

// a[i] for a lane-dependent i without dynamic register indexing
template <int N>
__device__ __forceinline__ float pick(const float (&a)[N], int i) {
  float r = a[0];
#pragma unroll
  for (int k = 1; k < N; ++k) r = (i == k) ? a[k] : r;
  return r;
}

// CTA that owns flattened unit t when T units are cut into n equal shares
// (share c covers [floor(c T / n), floor((c + 1) T / n))).
__device__ __forceinline__ long long owner_of(long long t, long long T, long long n) {
  return ((t + 1) * n - 1) / T;
}

template <int D, int GS, bool INT8>
__global__ void __launch_bounds__(kDecodeThreads)
    decode_kernel(const __grid_constant__ DecodeParams p) {
  using C = DecodeCfg<D, GS, INT8>;
  constexpr int W = kDecodeWarps;
  const float kNegInf = -INFINITY;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t *stages = smem;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kStagesBytes);
  float *sc_all = reinterpret_cast<float *>(smem + C::kStagesBytes + C::kBarBytes);
  float *mg = sc_all + W * kUnitRows * GS;
  int *misc = reinterpret_cast<int *>(mg + W * GS * (D + 2));
  int *pref = misc + C::kMiscBytes / 4;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int B = p.n_seq;
  const int spu = p.n_kvh * p.n_sub;
  const long long cap = (long long)p.max_pages * p.page_size;

  // ---- units per sequence and their prefix sums (shared memory) ----------
  {
    const int chunk = (B + kDecodeThreads - 1) / kDecodeThreads;
    const int b0 = min(B, tid * chunk), b1 = min(B, b0 + chunk);
    int local = 0;
    for (int b = b0; b < b1; ++b) local += units_of(p.seq_lens[b], cap);
    int incl = local;
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, m);
      if (lane >= m) incl += v;
    }
    if (lane == 31) misc[warp] = incl;
    __syncthreads();
    int run = incl - local, total = 0;
    for (int w = 0; w < W; ++w) {
      if (w < warp) run += misc[w];
      total += misc[w];
    }
    for (int b = b0; b < b1; ++b) {
      pref[b] = run;
      run += units_of(p.seq_lens[b], cap);
    }
    if (tid == 0) pref[B] = total;
    if (tid == 0) {
      for (int s = 0; s < W * C::kSW; ++s) mbar_init(&bars[s], 1);
      fence_barrier_init();
    }
    __syncthreads();
  }
  const long long T = (long long)spu * pref[B];
  if (T == 0) return;
  const long long n_active = min((long long)gridDim.x, max(1LL, (T + p.min_units - 1) / p.min_units));
  const int c = blockIdx.x;
  if (c >= n_active) return;
  const long long t0 = (long long)c * T / n_active;
  const long long t1 = (long long)(c + 1) * T / n_active;

  // everything below reads what the RoPE/append grid wrote
  pdl_wait_primary();

  const long long span = t1 - t0;
  const int count_w = span > warp ? (int)((span - warp - 1) / W + 1) : 0;
  const int cc = lane % C::kLPR, rg = lane / C::kLPR;
  const uint64_t pol = l2_evict_first_policy();

  // sequence containing flattened unit t0 (binary search on the prefix sums)
  int start_b;
  {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if ((long long)spu * pref[mid] <= t0) lo = mid; else hi = mid - 1;
    }
    start_b = lo;
  }

  // ---- producer side (lane 0 of each warp) --------------------------------
  int ib = start_b;  // issue cursor
  auto issue = [&](int i) {
    const long long t = t0 + warp + (long long)i * W;
    while ((long long)spu * pref[ib + 1] <= t) ++ib;
    const int units = pref[ib + 1] - pref[ib];
    const long long r = t - (long long)spu * pref[ib];
    const int si = (int)(r / units), u = (int)(r % units);
    const int j = si / p.n_sub;
    const int tok = u * kUnitRows;
    const int page = p.block_table[(size_t)ib * p.max_pages + tok / p.page_size];
    const int st = warp * C::kSW + i % C::kSW;
    uint8_t *dst = stages + (size_t)st * C::kStage;
    if (page >= 0 && page < p.num_pages) {
      const size_t row = ((size_t)page * p.n_kvh + j) * p.page_size + tok % p.page_size;
      mbar_arrive_expect_tx(&bars[st], C::kStage);
      bulk_g2s(dst, static_cast<const uint8_t *>(p.k_pages) + row * D * C::kESize, C::kTile,
               &bars[st], pol);
      bulk_g2s(dst + C::kTile, static_cast<const uint8_t *>(p.v_pages) + row * D * C::kESize,
               C::kTile, &bars[st], pol);
      if constexpr (INT8) {
        bulk_g2s(dst + 2 * C::kTile, p.k_scales + row, C::kScaleBytes, &bars[st], pol);
        bulk_g2s(dst + 2 * C::kTile + C::kScaleBytes, p.v_scales + row, C::kScaleBytes,
                 &bars[st], pol);
      }
    } else {
      mbar_arrive(&bars[st]);  // nothing to copy: complete the phase at once
    }
  };
  int issued = 0;
  if (lane == 0) {
    const int n0 = min(C::kSW, count_w);
    for (int i = 0; i < n0; ++i) issue(i);
    issued = n0;
  }

  // ---- consumer side ---------------------------------------------------------
  float *sc = sc_all + warp * kUnitRows * GS;
  float *mg_m = mg + W * GS * D;
  float *mg_l = mg_m + W * GS;
  volatile int *flag = misc + 8;
  bool aborted = false;
  int consumed = 0;
  int cb = start_b;
  long long t = t0;
  while (t < t1) {
    while ((long long)spu * pref[cb + 1] <= t) ++cb;
    const int units = pref[cb + 1] - pref[cb];
    const long long base = (long long)spu * pref[cb];
    const int si = (int)((t - base) / units);
    const long long F = base + (long long)si * units, E = F + units;
    const long long e = min(t1, E);
    const int L = p.seq_lens[cb];
    const int j = si / p.n_sub, sub = si % p.n_sub;
    const int h0 = j * GS * p.n_sub + sub * GS;

    float q[GS][8];
    {
      const float *qp = p.qhat + ((size_t)cb * p.n_qh + h0) * D + cc * 8;
#pragma unroll
      for (int hh = 0; hh < GS; ++hh) {
        const float4 x0 = *reinterpret_cast<const float4 *>(qp + hh * D);
        const float4 x1 = *reinterpret_cast<const float4 *>(qp + hh * D + 4);
        q[hh][0] = x0.x; q[hh][1] = x0.y; q[hh][2] = x0.z; q[hh][3] = x0.w;
        q[hh][4] = x1.x; q[hh][5] = x1.y; q[hh][6] = x1.z; q[hh][7] = x1.w;
      }
    }
    float m[GS], acc[GS][8], ls[C::kHPL];
#pragma unroll
    for (int hh = 0; hh < GS; ++hh) {
      m[hh] = kNegInf;
#pragma unroll
      for (int k = 0; k < 8; ++k) acc[hh][k] = 0.f;
    }
#pragma unroll
    for (int k = 0; k < C::kHPL; ++k) ls[k] = 0.f;

    const long long rel = t - t0;
    long long tt = t + ((warp - rel) % W + W) % W;
    for (; tt < e; tt += W) {
      const int i = (int)((tt - t0 - warp) / W);
      const int st = warp * C::kSW + i % C::kSW;
      bool ok = false;
      if (!aborted) {
        ok = mbar_wait_bounded(&bars[st], (uint32_t)((i / C::kSW) & 1));
        ok = __all_sync(0xffffffffu, ok);  // one decision per warp
        if (!ok) {
          aborted = true;
          if (lane == 0) atomicOr(p.status, KVATTN_DEV_TIMEOUT);
        }
      }
      consumed = i + 1;
      const int tok0 = (int)(tt - F) * kUnitRows;
      const int page = p.block_table[(size_t)cb * p.max_pages + tok0 / p.page_size];
      const bool page_ok = page >= 0 && page < p.num_pages;
      if (!page_ok && lane == 0) atomicOr(p.status, KVATTN_DEV_BAD_PAGE);
      if (ok && page_ok) {
        const int nrows = min(kUnitRows, L + 1 - tok0);
        const uint8_t *Ks = stages + (size_t)st * C::kStage;
        const uint8_t *Vs = Ks + C::kTile;
        const float *kscl = reinterpret_cast<const float *>(Ks + 2 * C::kTile);
        const float *vscl = kscl + kUnitRows;

        // scores: partial dots of the lane's 8 elements, then the butterfly
        float part[C::kNV];
#pragma unroll
        for (int pp = 0; pp < C::kNPass; ++pp) {
          const int row = pp * C::kRPP + rg;
          float kf[8];
          load_row8<INT8>(Ks + ((size_t)row * D + cc * 8) * C::kESize, kf);
#pragma unroll
          for (int hh = 0; hh < GS; ++hh) {
            float s = q[hh][0] * kf[0];
#pragma unroll
            for (int k = 1; k < 8; ++k) s = fmaf(q[hh][k], kf[k], s);
            part[pp * GS + hh] = s;
          }
        }
        TransposeReduce<C::kNV, C::kLPR / 2>::run(part, lane);
#pragma unroll
        for (int i2 = 0; i2 < C::kNVL; ++i2) {
          const int idx = i2 + (cc * C::kNV) / C::kLPR;
          const int row = (idx / GS) * C::kRPP + rg;
          bool writer = true;
          if constexpr (C::kNV < C::kLPR) writer = (cc % (C::kLPR / C::kNV)) == 0;
          if (writer) {
            float s = part[i2];
            if constexpr (INT8) s *= kscl[row];
            sc[row * GS + idx % GS] = (row < nrows) ? s : kNegInf;
          }
        }
        __syncwarp();

        // online softmax over the 16 rows of the unit
        const int srow = lane & 15, half = lane >> 4;
        float lmx[C::kHPL];
#pragma unroll
        for (int k = 0; k < C::kHPL; ++k) {
          const int hh = half + 2 * k;
          float v = (hh < GS) ? sc[srow * GS + hh] : kNegInf;
#pragma unroll
          for (int msk = 8; msk >= 1; msk >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, msk));
          lmx[k] = v;
        }
        float alpha[GS];
#pragma unroll
        for (int hh = 0; hh < GS; ++hh) {
          const float tm = __shfl_sync(0xffffffffu, lmx[hh >> 1], (hh & 1) << 4);
          const float mn = fmaxf(m[hh], tm);
          alpha[hh] = (mn == kNegInf) ? 1.f : exp2f(m[hh] - mn);
          m[hh] = mn;
        }
#pragma unroll
        for (int k = 0; k < C::kHPL; ++k) {
          const int hh = half + 2 * k;
          if (hh < GS) {
            const float s = sc[srow * GS + hh];
            const float mh = pick(m, hh);
            const float pv = (mh == kNegInf) ? 0.f : exp2f(s - mh);
            ls[k] = ls[k] * pick(alpha, hh) + pv;
            if constexpr (INT8) sc[srow * GS + hh] = pv * vscl[srow];
            else sc[srow * GS + hh] = pv;
          }
        }
#pragma unroll
        for (int hh = 0; hh < GS; ++hh)
#pragma unroll
          for (int k = 0; k < 8; ++k) acc[hh][k] *= alpha[hh];
        __syncwarp();

        // weighted value sum
#pragma unroll
        for (int pp = 0; pp < C::kNPass; ++pp) {
          const int row = pp * C::kRPP + rg;
          if (row < nrows) {
            float pv[GS];
#pragma unroll
            for (int hh = 0; hh < GS; ++hh) pv[hh] = sc[row * GS + hh];
            float vf[8];
            load_row8<INT8>(Vs + ((size_t)row * D + cc * 8) * C::kESize, vf);
#pragma unroll
            for (int hh = 0; hh < GS; ++hh)
#pragma unroll
              for (int k = 0; k < 8; ++k) acc[hh][k] = fmaf(pv[hh], vf[k], acc[hh][k]);
          }
        }
      }
      __syncwarp();
      if (lane == 0 && !aborted && issued < count_w) {
        fence_proxy_async_smem();
        issue(issued);
        ++issued;
      }
    }

    // ---- end of this stream's share: warp states -> CTA state --------------
#pragma unroll
    for (int msk = C::kLPR; msk < 32; msk <<= 1)
#pragma unroll
      for (int hh = 0; hh < GS; ++hh)
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[hh][k] += __shfl_xor_sync(0xffffffffu, acc[hh][k], msk);
#pragma unroll
    for (int k = 0; k < C::kHPL; ++k)
#pragma unroll
      for (int msk = 8; msk >= 1; msk >>= 1) ls[k] += __shfl_xor_sync(0xffffffffu, ls[k], msk);
    if (lane < C::kLPR) {
#pragma unroll
      for (int hh = 0; hh < GS; ++hh) {
        float *dst = mg + (warp * GS + hh) * D + cc * 8;
        *reinterpret_cast<float4 *>(dst) = make_float4(acc[hh][0], acc[hh][1], acc[hh][2], acc[hh][3]);
        *reinterpret_cast<float4 *>(dst + 4) = make_float4(acc[hh][4], acc[hh][5], acc[hh][6], acc[hh][7]);
      }
    }
    if ((lane & 15) == 0) {
#pragma unroll
      for (int k = 0; k < C::kHPL; ++k) {
        const int hh = (lane >> 4) + 2 * k;
        if (hh < GS) mg_l[warp * GS + hh] = ls[k];
      }
    }
    if (lane == 0) {
#pragma unroll
      for (int hh = 0; hh < GS; ++hh) mg_m[warp * GS + hh] = m[hh];
    }
    named_barrier_sync(1, kDecodeThreads);

    const bool whole = (F >= t0) && (E <= t1);
    const int sid = cb * spu + si;
    __nv_bfloat16 *outp = p.out + ((size_t)cb * p.n_qh + h0) * D;
    float *rec = p.records + (size_t)(sid + c) * (GS * (D + 2));
    for (int idx = tid; idx < GS * D; idx += kDecodeThreads) {
      const int hh = idx / D, dd = idx % D;
      float M = kNegInf;
#pragma unroll
      for (int w = 0; w < W; ++w) M = fmaxf(M, mg_m[w * GS + hh]);
      float o = 0.f, l = 0.f;
      if (M != kNegInf) {
#pragma unroll
        for (int w = 0; w < W; ++w) {
          const float f = exp2f(mg_m[w * GS + hh] - M);
          o += f * mg[(w * GS + hh) * D + dd];
          l += f * mg_l[w * GS + hh];
        }
      }
      if (whole) {
        outp[hh * D + dd] = __float2bfloat16_rn(l > 0.f ? o / l : 0.f);
      } else {
        rec[hh * D + dd] = o;
        if (dd == 0) {
          rec[GS * D + hh] = M;
          rec[GS * D + GS + hh] = l;
        }
      }
    }
    if (!whole) {
      __threadfence();
      named_barrier_sync(1, kDecodeThreads);
      if (tid == 0) {
        const long long c0 = owner_of(F, T, n_active), c1 = owner_of(E - 1, T, n_active);
        const unsigned nseg = (unsigned)(c1 - c0 + 1);
        const unsigned old = atomicAdd(&p.counters[sid], 1u);
        flag[0] = (old == nseg - 1) ? 1 : 0;
        flag[1] = (int)c0;
        flag[2] = (int)nseg;
      }
      named_barrier_sync(1, kDecodeThreads);
      if (flag[0]) {
        __threadfence();
        const int c0 = flag[1], nseg = flag[2];
        const float *r0 = p.records + (size_t)(sid + c0) * (GS * (D + 2));
        for (int idx = tid; idx < GS * D; idx += kDecodeThreads) {
          const int hh = idx / D, dd = idx % D;
          float M = kNegInf;
          for (int s = 0; s < nseg; ++s)
            M = fmaxf(M, __ldcg(r0 + (size_t)s * GS * (D + 2) + GS * D + hh));
          float o = 0.f, l = 0.f;
          if (M != kNegInf) {
            for (int s = 0; s < nseg; ++s) {
              const float *rs = r0 + (size_t)s * GS * (D + 2);
              const float f = exp2f(__ldcg(rs + GS * D + hh) - M);
              o += f * __ldcg(rs + hh * D + dd);
              l += f * __ldcg(rs + GS * D + GS + hh);
            }
          }
          outp[hh * D + dd] = __float2bfloat16_rn(l > 0.f ? o / l : 0.f);
        }
      }
    }
    named_barrier_sync(1, kDecodeThreads);
    t = e;
  }

  // after a timeout, wait (bounded) for this warp's copies still in flight so
  // that no bulk copy lands in shared memory after the CTA has exited
  if (aborted && lane == 0) {
    for (int i = consumed; i < issued; ++i)
      (void)mbar_wait_bounded(&bars[warp * C::kSW + i % C::kSW], (uint32_t)((i / C::kSW) & 1));
  }
}

template <int D, int GS, bool INT8>
cudaError_t launch_decode_t(const DecodeParams &p, int grid, cudaStream_t stream,
                            int *ctas_per_sm, bool launch) {
  using C = DecodeCfg<D, GS, INT8>;
  auto kern = decode_kernel<D, GS, INT8>;
  const int smem = C::kFixedSmem + (int)align_up((size_t)(p.n_seq + 1) * 4, 16);
  // per-device set-up and occupancy are cached so that steady-state calls make
  // no CUDA queries (and can be captured into a CUDA graph)
  static std::mutex mu;
  static std::map<std::pair<int, int>, int> occupancy;  // (device, smem) -> CTAs/SM
  static std::set<int> configured;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (ctas_per_sm) {
    std::lock_guard<std::mutex> lock(mu);
    if (!configured.count(dev)) {
      err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::kFixedSmem + (KVATTN_MAX_SEQS + 1) * 4 + 16);
      if (err != cudaSuccess) return err;
      configured.insert(dev);
    }
    auto it = occupancy.find({dev, smem});
    if (it == occupancy.end()) {
      int n = 0;
      err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kDecodeThreads, smem);
      if (err != cudaSuccess) return err;
      it = occupancy.emplace(std::make_pair(dev, smem), n).first;
    }
    *ctas_per_sm = it->second;
  }
  if (!launch) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kDecodeThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace kvattn
