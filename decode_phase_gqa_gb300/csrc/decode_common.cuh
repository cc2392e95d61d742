// Pieces shared by the decode and combine kernels: the balanced work split
// over all (sequence, KV head, query-head group) streams, the fp32 RoPE angle
// reduction of the query, and PTX wrappers for asynchronous copies, TMA tensor
// copies and warp-level tensor-core operations.
#pragma once

#include <cuda.h>

#include "kvattn_internal.cuh"

namespace kvattn {

// floor(a / b) for 0 <= a < 2^31 and 1 <= b whose quotient is below 2^20:
// a quotient estimate from the fp32 reciprocal of b (relative error under
// 2^-21, so within one of the quotient) corrected on the remainder.  A few
// dependent instructions instead of the general integer division, which
// weighs on the latency-bound set-up of a small decode step.
__device__ __forceinline__ int div_small(int a, int b) {
  float rb;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(rb) : "f"((float)b));
  int q = (int)((float)a * rb);
  const long long r = (long long)a - (long long)q * b;
  q += (int)(r >= b) - (int)(r < 0);
  return q;
}

// T units cut into n equal shares: share c covers [begin(c), begin(c + 1)),
// begin(c) = floor(c T / n) = c q + floor(c r / n) with T = q n + r.  All in
// 32-bit integers (the host keeps T below 2^31 and n <= 4096, so c r < 2^24
// and its quotient by n is below 2^12): a 64-bit division is a long software
// routine on this GPU.
struct Split {
  int T, n, q, r;
  __device__ __forceinline__ Split(int T_, int n_) : T(T_), n(n_), q(T_ / n_), r(T_ - (T_ / n_) * n_) {}
  __device__ __forceinline__ int begin(int c) const { return c * q + div_small(c * r, n); }
  // share holding unit t (0 <= t < T): an fp32 estimate of t n / T, off by
  // at most one, corrected against the exact boundaries
  __device__ __forceinline__ int owner(int t) const {
    int c = min(n - 1, (int)((float)t * ((float)n / (float)T)));
    while (c > 0 && begin(c) > t) --c;
    while (c + 1 < n && begin(c + 1) <= t) ++c;
    return c;
  }
};

// 2^x and log2(x) from the special-function unit's approximations (relative
// error near 2^-22; subnormal arguments and results flush to zero; 2^-inf = 0)
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two int8 codes of `u` (bytes selected by `sel`, a prmt selector whose other
// nibbles pick 0x64) as an f16 pair.  The codes arrive with their sign bit
// flipped (x + 128, an unsigned byte b); 0x6400 | b is the f16 1024 + b, and
// subtracting 1152 leaves x exactly (the magic-number integer conversion).
__device__ __forceinline__ uint32_t codes_to_f16x2(uint32_t u_flipped, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(u_flipped), "r"(0x64646464u), "r"(sel));
  asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(r) : "r"(0x64806480u));
  return r;
}

// Two int8 codes of `u` as the f16 pair 1152 + x: the conversion above
// without its subtraction, for MMAs whose accumulators take the bias off
// (1152 times the sum of the other operand, formed by an MMA with the
// constant pair kF16x2_1152).
__device__ __forceinline__ uint32_t codes_biased_f16x2(uint32_t u_flipped, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(u_flipped), "r"(0x64646464u), "r"(sel));
  return r;
}
constexpr uint32_t kF16x2_1152 = 0x64806480u;  // the f16 pair (1152, 1152)

// a[i] for a lane-dependent i without dynamic register indexing
template <int N>
__device__ __forceinline__ float pick(const float (&a)[N], int i) {
  float r = a[0];
#pragma unroll
  for (int k = 1; k < N; ++k) r = (i == k) ? a[k] : r;
  return r;
}

// ---- work split --------------------------------------------------------------
// Units per sequence and their prefix sums into shared memory (pref[0..B]);
// T = units over all streams (below 2^31: the host bounds it by the block
// table's capacity).  Returns false when there is nothing to do.
// `scratch` holds at least kThreads / 32 ints.  All threads of the CTA call it;
// with `report`, out-of-range lengths set KVATTN_DEV_BAD_LEN in the status word.
template <int kThreads>
__device__ __forceinline__ bool plan_units(const DecodeParams &p, int *pref, int *scratch,
                                           int &T, int *lens = nullptr,
                                           int *poss = nullptr, bool report = false) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = p.n_seq;
  const int spu = p.n_kvh * p.n_sub;
  const long long cap = (long long)p.max_pages * p.page_size;
  const int chunk = (B + kThreads - 1) / kThreads;
  const int b0 = min(B, tid * chunk), b1 = min(B, b0 + chunk);
  int local = 0;
  bool bad = false;
#pragma unroll 1
  for (int b = b0; b < b1; ++b) {
    const int L = __ldg(p.seq_lens + b);
    if (poss) poss[b] = __ldg(p.positions + b);  // in flight with the length
    const int n = units_of(L, cap);
    bad |= n == 0 && report;  // only an out-of-range length spans no unit
    local += n;
    if (lens) lens[b] = L;
  }
  if (bad) atomicOr(p.status, KVATTN_DEV_BAD_LEN);
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
#pragma unroll 1
  for (int b = b0; b < b1; ++b) {
    pref[b] = run;
    run += units_of(lens ? lens[b] : __ldg(p.seq_lens + b), cap);
  }
  if (tid == 0) pref[B] = total;
  __syncthreads();
  T = spu * pref[B];
  return T > 0;
}

// Layers.  A call may decode L layer caches that share the lengths,
// positions and block table (a layer-major batch): layer l's streams follow
// layer l - 1's in the unit list.  Sequence b of layer l is the virtual
// sequence v = l B + b; its queries, new rows, outputs and partial records are
// row v of the layer-major arrays, its pages those of layer l's pool.
//
// The split actually used: a warp share is an equal part of a weighted unit
// list, in which every unit weighs 4 and every stream weighs `sc` more (its
// fixed costs: the query set-up at its start, the new token's row at its end),
// placed after its last unit.  Unit t of stream s (s = v spu + si) sits at
// weighted position 4 t + sc s; a layer is XL = 4 TL + sc B spu long (TL: its
// units) and the list L XL (the host keeps it below 2^31).  Share c holds the
// units whose positions fall in [split.begin(c), split.begin(c + 1)); its
// unit range is [first_unit(split.begin(c)), first_unit(split.begin(c + 1))).
struct WeightedSplit {
  const int *pref;  // units per stream, prefix over the sequences of a layer
  int B, spu, sc, TL, XL, L;
  Split split;
  __device__ __forceinline__ WeightedSplit(const int *pref_, int B_, int spu_, int sc_, int TL_,
                                           int L_, int n)
      : pref(pref_), B(B_), spu(spu_), sc(sc_), TL(TL_), XL(4 * TL_ + sc_ * B_ * spu_), L(L_),
        split(L_ * (4 * TL_ + sc_ * B_ * spu_), n) {}
  // weighted position of sequence b's first stream within its layer
  __device__ __forceinline__ int seq_pos(int b) const { return 4 * spu * pref[b] + sc * spu * b; }
  // First unit whose weighted position is >= y (L TL when there is none) and
  // its virtual sequence *v (the sequence of the unit; L B - 1 when there is
  // none), found by one lane: the layer, then a binary search for the last
  // sequence of the layer starting at or before y, the stream and unit inside
  // it, and a second binary search that moves past sequences without units
  // (the unit then belongs to the next sequence that has some).  LAYERED:
  // whether the list may hold more than one layer (else L is 1).
  template <bool LAYERED>
  __device__ __forceinline__ int first_unit(int y, int *v) const {
    if (y >= split.T) {
      *v = L * B - 1;
      return L * TL;
    }
    const int l = (LAYERED && y >= XL) ? div_small(y, XL) : 0;  // (l < L <= 1024)
    y -= l * XL;
    int lo = 0, hi = B;  // seq_pos(lo) <= y; every sequence from hi on starts after y
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (seq_pos(mid) <= y)
        lo = mid;
      else
        hi = mid;
    }
    const int u = pref[lo + 1] - pref[lo];
    const int ws = 4 * u + sc;  // > 0: y lies inside sequence lo's streams
    const int off = y - seq_pos(lo);
    const int si = div_small(off, ws), rem = off - si * ws;  // (off < spu ws: si < spu)
    const int t = spu * pref[lo] + si * u + min(u, (rem + 3) >> 2);
    int bl = lo, bh = B;  // the last sequence whose first unit is at or before t
    while (bh - bl > 1) {
      const int mid = (bl + bh) >> 1;
      if (spu * pref[mid] <= t)
        bl = mid;
      else
        bh = mid;
    }
    *v = l * B + bl;
    return l * TL + t;
  }
  // first_unit for a batch of at most 32 sequences, by the whole warp at
  // once: lane b holds pref[b] (pl; any value for b >= B), and the two
  // searches are ballots over the sequences (seq_pos and pref are
  // nondecreasing, so the sequences at or before a position are a prefix).
  template <bool LAYERED>
  __device__ __forceinline__ int first_unit_warp(int y, int *v, int lane, int pl) const {
    if (y >= split.T) {
      *v = L * B - 1;
      return L * TL;
    }
    const int l = (LAYERED && y >= XL) ? div_small(y, XL) : 0;
    y -= l * XL;
    const bool in = lane < B;
    const int lo = __popc(__ballot_sync(0xffffffffu, in && 4 * spu * pl + sc * spu * lane <= y)) - 1;
    const int p0 = __shfl_sync(0xffffffffu, pl, lo);
    const int u = pref[lo + 1] - p0;
    const int ws = 4 * u + sc;
    const int off = y - (4 * spu * p0 + sc * spu * lo);
    const int si = div_small(off, ws), rem = off - si * ws;
    const int t = spu * p0 + si * u + min(u, (rem + 3) >> 2);
    const int bl = __popc(__ballot_sync(0xffffffffu, in && spu * pl <= t)) - 1;
    *v = l * B + bl;
    return l * TL + t;
  }
  // Unit range [*t0, *t1) of share c and the virtual sequences of its ends,
  // for the whole warp: up to 32 sequences by ballots (both ends in turn),
  // else even lanes search the start and odd lanes the end, at once.
  template <bool LAYERED>
  __device__ __forceinline__ void share_bounds(int c, int lane, int *t0, int *b0, int *t1,
                                               int *b1) const {
    if (B <= 32) {
      const int pl = lane < B ? pref[lane] : 0;
      *t0 = first_unit_warp<LAYERED>(split.begin(c), b0, lane, pl);
      *t1 = first_unit_warp<LAYERED>(split.begin(c + 1), b1, lane, pl);
      return;
    }
    int b = 0;
    const int t = first_unit<LAYERED>(split.begin(c + (lane & 1)), &b);
    *t0 = __shfl_sync(0xffffffffu, t, 0);
    *b0 = __shfl_sync(0xffffffffu, b, 0);
    *t1 = __shfl_sync(0xffffffffu, t, 1);
    *b1 = __shfl_sync(0xffffffffu, b, 1);
  }
  // share holding unit t of stream sid
  __device__ __forceinline__ int owner(int t, int sid) const { return split.owner(4 * t + sc * sid); }
};

// Number of warp shares a step's weighted unit list (X = 4 per unit plus the
// stream costs) is cut into, for a grid of n_warps warps.  A share's time is
// set by the units it streams one after another, so a small step takes
// shares of at most 3 units (X / 12 of them) when that keeps at least half of
// the warps free (they help the appending warps; the shares are spread over
// the CTAs), else of at most 4 units (X / 16), a unit weighing 4: more shares
// than that would only add partial states to merge.  The decode and combine
// kernels both call this.
__device__ __forceinline__ int warp_shares(int X, int n_warps) {
  const int n3 = X / 12 + (X % 12 != 0), n4 = X / 16 + (X % 16 != 0);  // (X may be near 2^31)
  if (2 * n3 <= n_warps) return max(1, n3);
  return max(1, min(n_warps, n4));
}

// Position of flattened unit t: virtual sequence (cursor v, advanced
// monotonically), its layer and sequence within the layer, stream within the
// sequence and unit within the stream (TL: units per layer).
struct UnitPos {
  int v, l, b, si, u, units;
  int first;  // flattened index of the stream's first unit
};

template <bool LAYERED>  // (else l is 0 and v is b)
__device__ __forceinline__ UnitPos locate_unit(int t, int &v, const int *pref, int spu, int B,
                                               int TL) {
  int l = 0, b = v;
  if (LAYERED && v >= B) {
    l = div_small(v, B);  // (l < L <= 1024)
    b = v - l * B;
  }
  while ((LAYERED ? l * TL : 0) + spu * pref[b + 1] <= t) {  // unit t lies past sequence (l, b)
    ++b;
    if (LAYERED && b == B) {
      b = 0;
      ++l;
    }
  }
  v = l * B + b;
  UnitPos r;
  r.v = v;
  r.l = l;
  r.b = b;
  r.units = pref[b + 1] - pref[b];
  const int off = t - ((LAYERED ? l * TL : 0) + spu * pref[b]);
  r.si = div_small(off, r.units);  // (the stream within the sequence: below spu)
  r.u = off - r.si * r.units;
  r.first = t - r.u;
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

// block-table entry (physical page within its layer's pool, not yet
// range-checked) of flattened unit t (cursor v advanced monotonically)
template <bool LAYERED>
__device__ __forceinline__ int page_raw_of_unit(const DecodeParams &p, const int *pref, int spu,
                                                int TL, int t, int &v) {
  const UnitPos up = locate_unit<LAYERED>(t, v, pref, spu, p.n_seq, TL);
  return __ldg(p.block_table + (size_t)up.b * p.max_pages + (up.u >> p.unit_shift));
}

// 16-byte asynchronous global -> shared copy (no register staging)
__device__ __forceinline__ void cp_async_16(void *dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src)
               : "memory");
}
// make `bar` track this thread's earlier cp.async copies: its pending count
// is raised now and lowered when they have landed
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t *bar) {
  asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
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
