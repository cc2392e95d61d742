// Pieces shared by the decode kernels: the balanced work split over all
// (sequence, KV head, query-head group) streams, the CTA-level softmax-state
// merge and the last-arriver log-sum-exp merge of split streams, and PTX
// wrappers for TMA tensor copies and warp-level tensor-core operations.
#pragma once

#include <cuda.h>

#include "kvattn_internal.cuh"

namespace kvattn {

// CTA that owns flattened unit t when T units are cut into n equal shares
// (share c covers [floor(c T / n), floor((c + 1) T / n))).
__device__ __forceinline__ long long owner_of(long long t, long long T, long long n) {
  return ((t + 1) * n - 1) / T;
}

// a[i] for a lane-dependent i without dynamic register indexing
template <int N>
__device__ __forceinline__ float pick(const float (&a)[N], int i) {
  float r = a[0];
#pragma unroll
  for (int k = 1; k < N; ++k) r = (i == k) ? a[k] : r;
  return r;
}

// ---- work split --------------------------------------------------------------
struct Share {
  long long T;         // units over all streams
  long long n_active;  // CTAs with work
  long long t0, t1;    // this CTA's units [t0, t1)
  int start_b;         // sequence holding unit t0
};

// Units per sequence and their prefix sums into shared memory (pref[0..B]);
// T = units over all streams.  Returns false when there is nothing to do.
// `scratch` holds at least kThreads / 32 ints.  All threads of the CTA call it.
template <int kThreads>
__device__ __forceinline__ bool plan_units(const DecodeParams &p, int *pref, int *scratch,
                                           long long &T, int *lens = nullptr,
                                           int *poss = nullptr) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = p.n_seq;
  const int spu = p.n_kvh * p.n_sub;
  const long long cap = (long long)p.max_pages * p.page_size;
  const int chunk = (B + kThreads - 1) / kThreads;
  const int b0 = min(B, tid * chunk), b1 = min(B, b0 + chunk);
  int local = 0;
  for (int b = b0; b < b1; ++b) local += units_of(__ldg(p.seq_lens + b), cap);
  int incl = local;
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, m);
    if (lane >= m) incl += v;
  }
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  int run = incl - local, total = 0;
  for (int w = 0; w < kThreads / 32; ++w) {
    if (w < warp) run += scratch[w];
    total += scratch[w];
  }
  for (int b = b0; b < b1; ++b) {
    const int L = __ldg(p.seq_lens + b);
    pref[b] = run;
    run += units_of(L, cap);
    if (lens) lens[b] = L;
    if (poss) poss[b] = __ldg(p.positions + b);
  }
  if (tid == 0) pref[B] = total;
  __syncthreads();
  T = (long long)spu * pref[B];
  return T > 0;
}

// Sequence holding flattened unit t (binary search on the prefix sums).
__device__ __forceinline__ int seq_of_unit(long long t, const int *pref, int B, int spu) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((long long)spu * pref[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// CTA-level share of the flattened unit list (one share per CTA).
template <int kThreads>
__device__ __forceinline__ bool plan_share(const DecodeParams &p, int *pref, int *scratch,
                                           Share &sh) {
  if (!plan_units<kThreads>(p, pref, scratch, sh.T)) return false;
  sh.n_active = min((long long)min((int)gridDim.x, p.n_shares),
                    max(1LL, (sh.T + p.min_units - 1) / p.min_units));
  if ((long long)blockIdx.x >= sh.n_active) return false;
  sh.t0 = (long long)blockIdx.x * sh.T / sh.n_active;
  sh.t1 = (long long)(blockIdx.x + 1) * sh.T / sh.n_active;
  sh.start_b = seq_of_unit(sh.t0, pref, p.n_seq, p.n_kvh * p.n_sub);
  return true;
}

// Position of flattened unit t: sequence (cursor b, advanced monotonically),
// stream within the sequence and unit within the stream.
struct UnitPos {
  int b, si, u, units;
  long long first;  // flattened index of the stream's first unit
};

__device__ __forceinline__ UnitPos locate_unit(long long t, int &b, const int *pref, int spu) {
  while ((long long)spu * pref[b + 1] <= t) ++b;
  UnitPos r;
  r.b = b;
  r.units = pref[b + 1] - pref[b];
  const long long base = (long long)spu * pref[b];
  r.si = (int)((t - base) / r.units);
  r.u = (int)((t - base) % r.units);
  r.first = base + (long long)r.si * r.units;
  return r;
}

// ---- RoPE angles of the query, fp32 only -----------------------------------------
// Fractional part, in [-0.5, 0.5], of pos * g turns, g = g.x + g.y (fp32 head
// and remainder).  The position is split into a multiple of 4096 and a
// remainder (both exact in fp32), each product is split into its rounded value
// and exact rounding error with an FMA, and the fractional part of every piece
// is taken exactly (x - rint(x) is exact in binary floating point) before the
// pieces are added: the result is accurate to about 1e-7 turns for positions
// below 2^20, without any double-precision arithmetic.
__device__ __forceinline__ float frac_turns(int pos, float2 g) {
  const float ph = (float)(pos & ~0xfff), pl = (float)(pos & 0xfff);
  const float a = ph * g.x, ae = fmaf(ph, g.x, -a);
  const float b = pl * g.x, be = fmaf(pl, g.x, -b);
  float t = (a - rintf(a)) + (ae - rintf(ae));
  t += (b - rintf(b)) + (be - rintf(be));
  t -= rintf(t);
  const float c = (float)pos * g.y;
  t += c - rintf(c);
  return t - rintf(t);
}

// ---- queries ----------------------------------------------------------------------
// Rotated queries of one stream's GS heads, multiplied by scale * log2(e), into
// shared memory qs[GS][D] (fp32), using all kThreads threads of the CTA; cs
// holds D/2 float2.  The angles come from frac_turns and sincospif: the query
// needs fp32 accuracy only, the bit-exact recipe applies to the stored key.
template <int D, int GS, int kThreads>
__device__ __forceinline__ void stream_queries(const DecodeParams &p, int b, int h0, float *qs,
                                               float2 *cs) {
  constexpr int H = D / 2;
  constexpr int NP = (GS * H + kThreads - 1) / kThreads;  // pairs per thread
  const int tid = threadIdx.x;
  const __nv_bfloat16 *qb = p.q + ((size_t)b * p.n_qh + h0) * D;
  float lo[NP], hi[NP];
#pragma unroll
  for (int k = 0; k < NP; ++k) {
    const int idx = tid + k * kThreads;
    if (idx < GS * H) {
      const int hh = idx / H, i = idx % H;
      lo[k] = __bfloat162float(qb[hh * D + i]);
      hi[k] = __bfloat162float(qb[hh * D + i + H]);
    }
  }
  if (tid < H) {
    float c = 1.f, sn = 0.f;
    if (p.use_rope) sincospif(2.f * frac_turns(__ldg(p.positions + b), p.turns[tid]), &sn, &c);
    cs[tid] = make_float2(c, sn);
  }
  named_barrier_sync(1, kThreads);
#pragma unroll
  for (int k = 0; k < NP; ++k) {
    const int idx = tid + k * kThreads;
    if (idx < GS * H) {
      const int hh = idx / H, i = idx % H;
      const float2 r = cs[i];
      qs[hh * D + i] = (lo[k] * r.x - hi[k] * r.y) * p.qscale;
      qs[hh * D + i + H] = (hi[k] * r.x + lo[k] * r.y) * p.qscale;
    }
  }
  named_barrier_sync(1, kThreads);
}

// ---- merges ---------------------------------------------------------------------
// The CTA's warps have left their states in shared memory: acc at
// mg[(w*GS + hh)*D + d], m at mg_m[w*GS + hh], l at mg_l[w*GS + hh] (m in log2
// units, acc and l relative to 2^m).  Combine them; a stream wholly inside this
// CTA is written to `out`, otherwise a record (acc[GS][D], m[GS], l[GS]) goes
// to the workspace and the last CTA to arrive merges all records of the stream.
template <int D, int GS, int W, int kThreads>
__device__ __forceinline__ void finish_stream(const DecodeParams &p, const Share &sh,
                                              const float *mg, const float *mg_m,
                                              const float *mg_l, int *flags, float *red,
                                              long long F, long long E, int b, int sid,
                                              int h0) {
  const float kNegInf = -INFINITY;
  const int tid = threadIdx.x;
  const bool whole = (F >= sh.t0) && (E <= sh.t1);
  __nv_bfloat16 *outp = p.out + ((size_t)b * p.n_qh + h0) * D;
  constexpr int RS = record_floats(GS, D);  // floats per record
  float *rec = p.records + (size_t)(sid + blockIdx.x) * RS;
  for (int idx = tid; idx < GS * D; idx += kThreads) {
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
  if (whole) return;
  __threadfence();
  named_barrier_sync(1, kThreads);
  if (tid == 0) {
    const long long c0 = owner_of(F, sh.T, sh.n_active), c1 = owner_of(E - 1, sh.T, sh.n_active);
    const unsigned nseg = (unsigned)(c1 - c0 + 1);
    const unsigned old = atomicAdd(&p.counters[sid], 1u);
    flags[0] = (old == nseg - 1) ? 1 : 0;
    // every share of the stream has arrived: leave the counter at zero for the
    // next call (the workspace starts zeroed)
    if (old == nseg - 1) p.counters[sid] = 0u;
    flags[1] = (int)c0;
    flags[2] = (int)nseg;
  }
  named_barrier_sync(1, kThreads);
  if (!flags[0]) return;
  __threadfence();
  const int c0 = flags[1], nseg = flags[2];
  const float *r0 = p.records + (size_t)(sid + c0) * RS;
  // pass 1: per-head maximum and normaliser over the records (block reduction)
  float mloc[GS];
#pragma unroll
  for (int hh = 0; hh < GS; ++hh) mloc[hh] = kNegInf;
  for (int s = tid; s < nseg; s += kThreads)
#pragma unroll
    for (int hh = 0; hh < GS; ++hh)
      mloc[hh] = fmaxf(mloc[hh], __ldcg(r0 + (size_t)s * RS + GS * D + hh));
  const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
  for (int hh = 0; hh < GS; ++hh) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) mloc[hh] = fmaxf(mloc[hh], __shfl_xor_sync(0xffffffffu, mloc[hh], m));
    if (lane == 0) red[warp * GS + hh] = mloc[hh];
  }
  named_barrier_sync(1, kThreads);
  float M[GS];
#pragma unroll
  for (int hh = 0; hh < GS; ++hh) {
    M[hh] = kNegInf;
    for (int w = 0; w < kThreads / 32; ++w) M[hh] = fmaxf(M[hh], red[w * GS + hh]);
  }
  float lsum[GS];
#pragma unroll
  for (int hh = 0; hh < GS; ++hh) lsum[hh] = 0.f;
  for (int s = tid; s < nseg; s += kThreads) {
    const float *rs = r0 + (size_t)s * RS;
#pragma unroll
    for (int hh = 0; hh < GS; ++hh) {
      const float ms = __ldcg(rs + GS * D + hh);
      if (M[hh] != kNegInf) lsum[hh] += exp2f(ms - M[hh]) * __ldcg(rs + GS * D + GS + hh);
    }
  }
  named_barrier_sync(1, kThreads);  // everyone has read the maxima
#pragma unroll
  for (int hh = 0; hh < GS; ++hh) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) lsum[hh] += __shfl_xor_sync(0xffffffffu, lsum[hh], m);
    if (lane == 0) red[warp * GS + hh] = lsum[hh];
  }
  named_barrier_sync(1, kThreads);
  // pass 2: each thread owns 4 consecutive output elements of one head
  for (int q4 = tid; q4 < GS * D / 4; q4 += kThreads) {
    const int hh = (q4 * 4) / D;
    float L = 0.f;
    for (int w = 0; w < kThreads / 32; ++w) L += red[w * GS + hh];
    const float Mh = pick(M, hh);
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    if (Mh != kNegInf) {
      int s = 0;
      for (; s + 4 <= nseg; s += 4) {
        float f[4];
        float4 a[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float *rs = r0 + (size_t)(s + k) * RS;
          f[k] = __ldcg(rs + GS * D + hh);
          a[k] = __ldcg(reinterpret_cast<const float4 *>(rs) + q4);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float e = exp2f(f[k] - Mh);
          o.x += e * a[k].x; o.y += e * a[k].y; o.z += e * a[k].z; o.w += e * a[k].w;
        }
      }
      for (; s < nseg; ++s) {
        const float *rs = r0 + (size_t)s * RS;
        const float e = exp2f(__ldcg(rs + GS * D + hh) - Mh);
        const float4 a = __ldcg(reinterpret_cast<const float4 *>(rs) + q4);
        o.x += e * a.x; o.y += e * a.y; o.z += e * a.z; o.w += e * a.w;
      }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    __nv_bfloat162 lo = __floats2bfloat162_rn(o.x * inv, o.y * inv);
    __nv_bfloat162 hi2 = __floats2bfloat162_rn(o.z * inv, o.w * inv);
    __nv_bfloat162 *dst = reinterpret_cast<__nv_bfloat162 *>(outp + q4 * 4);
    dst[0] = lo;
    dst[1] = hi2;
  }
}

// physical page of flattened unit t (cursor b advanced monotonically), or -1
// when the block-table entry is out of range
__device__ __forceinline__ int page_of_unit(const DecodeParams &p, const int *pref, int spu,
                                            long long t, int &b) {
  const UnitPos up = locate_unit(t, b, pref, spu);
  const int page =
      __ldg(p.block_table + (size_t)up.b * p.max_pages + (up.u * kUnitRows) / p.page_size);
  return (page >= 0 && page < p.num_pages) ? page : -1;
}

// 16-byte asynchronous global -> shared copy (no register staging)
__device__ __forceinline__ void cp_async_16(void *dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// ---- TMA tensor copies and warp-level tensor-core operations -------------------
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y,
                                            uint64_t *bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// D (16x8 fp32) += A (16x16 bf16, row) * B (16x8 bf16, col)
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// transpose of an 8x8 b16 matrix held in the accumulator-style fragment
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

}  // namespace kvattn
