// Split-KV flash-decoding kernel, CUDA-core inner loop (used for the int8 KV
// cache; the bf16 cache uses the tensor-core kernel of decode_mma.cuh).
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

#include "decode_common.cuh"

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
  static constexpr int kScBytes = kDecodeWarps * kUnitRows * GS * 4;
  static constexpr int kMergeBytes = kDecodeWarps * GS * (D + 3) * 4;  // acc, m, l, reduction
  static constexpr int kMiscBytes = 64;
  // stages per warp: as many as fit a 75 KB CTA (3 CTAs per SM) next to the
  // other buffers and a 1 KB allowance for the per-sequence prefix sums
  static constexpr int kOther = kDecodeWarps * 8 * 8 + kScBytes + kMergeBytes + kMiscBytes;
  static constexpr int kSWFit = (kCtaSmemBudget - kOther - 1024) / (kDecodeWarps * kStage);
  static constexpr int kSW = kSWFit > 8 ? 8 : kSWFit;
  static constexpr int kStagesBytes = kDecodeWarps * kSW * kStage;
  static constexpr int kBarBytes = kDecodeWarps * kSW * 8;
  static constexpr int kFixedSmem = kStagesBytes + kBarBytes + kScBytes + kMergeBytes + kMiscBytes;
  // the rotated queries [GS][D] and cos/sin [D/2] of a stream's start share
  // the merge area, which is only used at the stream's end
  static_assert(GS * D * 4 + (D / 2) * 8 <= kDecodeWarps * GS * D * 4, "query buffers");
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
  float *mg_m = mg + W * GS * D;
  float *mg_l = mg_m + W * GS;
  float *red = mg_l + W * GS;
  int *misc = reinterpret_cast<int *>(red + W * GS);
  int *pref = misc + C::kMiscBytes / 4;
  float *qs = mg;
  float2 *cs = reinterpret_cast<float2 *>(qs + GS * D);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int spu = p.n_kvh * p.n_sub;
  Share sh;
  if (!plan_share<kDecodeThreads>(p, pref, misc, sh)) return;
  if (tid == 0) {
    for (int s = 0; s < W * C::kSW; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
  }
  __syncthreads();
  const long long t0 = sh.t0, t1 = sh.t1;

  const long long span = t1 - t0;
  const int count_w = span > warp ? (int)((span - warp - 1) / W + 1) : 0;
  const int cc = lane % C::kLPR, rg = lane / C::kLPR;
  const uint64_t pol = l2_evict_first_policy();

  // ---- producer side (lane 0 of each warp) --------------------------------
  // Only the last unit of a stream holds the token the append grid writes in
  // this step: wait for that grid before the first such unit.
  int ib = sh.start_b;  // issue cursor
  bool appended_visible = false;
  auto issue = [&](int i) {
    const long long t = t0 + warp + (long long)i * W;
    const UnitPos up = locate_unit(t, ib, pref, spu);
    if (up.u == up.units - 1 && !appended_visible) {
      pdl_wait_primary();
      appended_visible = true;
    }
    const int j = up.si / p.n_sub;
    const int tok = up.u * kUnitRows;
    const int page = __ldg(p.block_table + (size_t)up.b * p.max_pages + tok / p.page_size);
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
    for (; issued < min(C::kSW, count_w); ++issued) issue(issued);
  }

  // ---- consumer side ---------------------------------------------------------
  float *sc = sc_all + warp * kUnitRows * GS;
  bool aborted = false;
  int consumed = 0;
  int cb = sh.start_b;
  long long t = t0;
  while (t < t1) {
    const UnitPos sp = locate_unit(t, cb, pref, spu);
    const int si = sp.si;
    const long long F = sp.first, E = F + sp.units;
    const long long e = min(t1, E);
    const int L = __ldg(p.seq_lens + cb);
    const int j = si / p.n_sub, sub = si % p.n_sub;
    const int h0 = j * GS * p.n_sub + sub * GS;

    stream_queries<D, GS, kDecodeThreads>(p, cb, h0, qs, cs);
    float q[GS][8];
#pragma unroll
    for (int hh = 0; hh < GS; ++hh) {
      const float4 x0 = *reinterpret_cast<const float4 *>(qs + hh * D + cc * 8);
      const float4 x1 = *reinterpret_cast<const float4 *>(qs + hh * D + cc * 8 + 4);
      q[hh][0] = x0.x; q[hh][1] = x0.y; q[hh][2] = x0.z; q[hh][3] = x0.w;
      q[hh][4] = x1.x; q[hh][5] = x1.y; q[hh][6] = x1.z; q[hh][7] = x1.w;
    }
    named_barrier_sync(1, kDecodeThreads);  // queries read: the merge area is free again
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

    finish_stream<D, GS, W, kDecodeThreads>(p, sh, mg, mg_m, mg_l, misc + 8, red, F, E, cb,
                                            cb * spu + si, h0);
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
