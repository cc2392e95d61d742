// Combine kernel: log-sum-exp merge of the streams the decode kernel's work
// split cut across warp shares (second launch of a step).
//
// A split stream leaves one partial record (acc[GS][d] relative to 2^m,
// m[GS], l[GS]; log2 units) per share it touches, in consecutive slots.  This
// kernel recomputes the decode kernel's split from the lengths and merges the
// records ("Qwen3-8B inference engine from scratch in C++/CUDA", section
// 4.4.1: the blockwise softmax recombines its blocks by rescaling with the
// running maximum):
//   M = max_r m_r,  L = sum_r 2^(m_r - M) l_r,  out = sum_r 2^(m_r - M) acc_r / L.
// Two CTAs per SM at most; CTA c takes items c, c + gridDim.x, ... and lists
// the merges to do while the decode grid still runs, so that only the record
// loads remain after the wait.  A thread merges the records of one float4
// column eight at a time (their largest maximum first, then the eight weights
// at once, so no exponential waits on another);
// a stream cut into many shares gives each column several record lanes,
// merged in shared memory, and spreads its columns over several CTAs.
// The kernel is launched as a programmatic dependent of the decode kernel and
// waits for it before reading anything the decode grid writes.
#include "decode_common.cuh"

namespace kvattn {

namespace {

constexpr int kCombineThreads = 256;

// running softmax state of one output column: max m, normaliser l (log2 units)
// and the four accumulator values, all relative to 2^m
struct ColState {
  float m, l;
  float4 o;
};

// Fold U states (m, l, a) into st at once: the batch's largest maximum first,
// then each weight 2^(m_u - M) on its own, so the exponentials do not wait on
// one another.  Empty slots carry m = -inf (weight 0, l = 0, a = 0).
template <int U>
__device__ __forceinline__ void absorb_batch(ColState &st, const float (&m)[U], const float (&l)[U],
                                             const float4 (&a)[U]) {
  float mb = st.m;
#pragma unroll
  for (int u = 0; u < U; ++u) mb = fmaxf(mb, m[u]);
  if (mb == -INFINITY) return;  // nothing but empty slots so far
  const float so = ex2_approx(st.m - mb);
  float ls = st.l * so;
  float4 o = make_float4(st.o.x * so, st.o.y * so, st.o.z * so, st.o.w * so);
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const float w = ex2_approx(m[u] - mb);
    ls = fmaf(l[u], w, ls);
    o.x = fmaf(a[u].x, w, o.x);
    o.y = fmaf(a[u].y, w, o.y);
    o.z = fmaf(a[u].z, w, o.z);
    o.w = fmaf(a[u].w, w, o.w);
  }
  st.m = mb;
  st.l = ls;
  st.o = o;
}

// Merge, by one thread, of column c of records r0 + r * RS for
// r = first, first + step, ... < nseg, eight loads in flight at a time.
template <int D, int GS>
__device__ __forceinline__ ColState merge_column(const float *r0, int first, int step, int nseg,
                                                 int c) {
  constexpr int RS = record_floats(GS, D);
  constexpr int U = 8;
  const int hc = (c * 4) / D;
  ColState st = {-INFINITY, 0.f, make_float4(0.f, 0.f, 0.f, 0.f)};
  for (int s0 = first; s0 < nseg; s0 += step * U) {
    float mm[U], ll[U];
    float4 a[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int r = s0 + u * step;
      if (r < nseg) {
        const float *rs = r0 + (size_t)r * RS;
        a[u] = __ldcg(reinterpret_cast<const float4 *>(rs) + c);
        mm[u] = __ldcg(rs + GS * D + hc);
        ll[u] = __ldcg(rs + GS * D + GS + hc);
      } else {
        mm[u] = -INFINITY;
        ll[u] = 0.f;
        a[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    absorb_batch<U>(st, mm, ll, a);
  }
  return st;
}

__device__ __forceinline__ void store_column(__nv_bfloat16 *dst4, const ColState &st) {
  const float inv = st.l > 0.f ? 1.f / st.l : 0.f;
  __nv_bfloat162 *dst = reinterpret_cast<__nv_bfloat162 *>(dst4);
  dst[0] = __floats2bfloat162_rn(st.o.x * inv, st.o.y * inv);
  dst[1] = __floats2bfloat162_rn(st.o.z * inv, st.o.w * inv);
}

template <int D, int GS>
__global__ void __launch_bounds__(kCombineThreads, 2)
    combine_kernel(const __grid_constant__ DecodeParams p, int n_warps) {
  constexpr int RS = record_floats(GS, D);
  constexpr int NC = GS * D / 4;  // float4 columns of a record's accumulator
  static_assert(kCombineThreads % NC == 0, "columns must tile the CTA");
  static_assert((NC & (NC - 1)) == 0, "chunk sizes and record lanes are powers of two");
  constexpr int kGroups = kCombineThreads / NC;  // concurrent short merges per CTA
  // A stream of at most kShort shares is merged by a group of NC threads,
  // one column each, kGroups at a time and without CTA barriers.  A longer
  // one takes R record lanes per column, R = its shares / 8 rounded up to a
  // power of two, so that one batch of eight records per thread covers them;
  // its columns are then split into nch = NC R / (CTA threads) items (each of
  // at least kMinCols columns, which caps R at 16) that different CTAs merge.
  // (Four records a lane, twice the items, was slower on the Qwen3-shaped
  // batch: a CTA merges its long items one after another.)
  constexpr int kShort = 8;
  constexpr int kMinCols = 16 < NC ? 16 : NC;
  constexpr int kMaxChunks = NC / kMinCols;
  __shared__ ColState part[kCombineThreads];  // [record lane][column]
  __shared__ int4 list[kCombineThreads];      // (first record slot, chunk, log2 chunks, v)
  __shared__ int lh0[kCombineThreads];        // first query head
  __shared__ int lseg[kCombineThreads];
  __shared__ int n_list;
  __shared__ int scratch[32];
  extern __shared__ int pref[];  // [n_seq + 1]

  // the next call's decode grid may be placed now: it waits for this grid to
  // end before it touches global memory
  pdl_launch_dependents();
  const int tid = threadIdx.x;
  const int spu = p.n_kvh * p.n_sub;
  // The decode kernel's split, recomputed from the lengths while it runs:
  // the unit list of T units is cut into nwa warp shares (WeightedSplit), and
  // stream sid's records sit in slots sid + (its first share) onwards, one
  // per share.
  int TL = 0;  // units of one layer
  const bool any = plan_units<kCombineThreads>(p, pref, scratch, TL);
  const int nwa =
      any ? warp_shares(p.n_layers * (4 * TL + p.stream_cost * p.n_seq * spu), n_warps) : 1;
  const WeightedSplit split(pref, p.n_seq, spu, p.stream_cost, any ? TL : 1, p.n_layers, nwa);
  const int n_streams = p.n_layers * p.n_seq * spu;  // stream sid: virtual sequence sid / spu
  // item it: chunk it / n_streams of stream it % n_streams; CTA c takes
  // items c, c + gridDim.x, ...
  const int n_items = any ? n_streams * kMaxChunks : 0;
  const int stride = (int)gridDim.x * kCombineThreads;
  bool waited = false;
  for (int base = blockIdx.x; base < n_items; base += stride) {
    if (tid == 0) n_list = 0;
    __syncthreads();
    const int it = base + tid * (int)gridDim.x;
    if (it < n_items) {
      const int q = it / n_streams, sid = it - q * n_streams;
      const int v = sid / spu, si = sid % spu;
      const int l = v / p.n_seq, b = v - l * p.n_seq;
      const int units = pref[b + 1] - pref[b];
      if (units > 0) {
        const int F = l * TL + spu * pref[b] + si * units;
        const int w0 = split.owner(F, sid);
        const int nseg = split.owner(F + units - 1, sid) - w0 + 1;
        int R = 1;
        while (R * 8 < nseg) R *= 2;
        const int nch = nseg <= kShort ? 1 : max(1, min(kMaxChunks, NC * R / kCombineThreads));
        if (nseg > 1 && q < nch) {
          const int k = atomicAdd(&n_list, 1);
          list[k] = make_int4(sid + w0, q, __ffs(nch) - 1, v);  // (nch: a power of two)
          lseg[k] = nseg;
          lh0[k] = (si / p.n_sub) * GS * p.n_sub + (si % p.n_sub) * GS;
        }
      }
    }
    __syncthreads();
    if (!waited) {
      pdl_wait_primary();  // the decode grid's records are complete and visible
      waited = true;
    }
    // short merges: group gi = tid / NC takes entries gi, gi + kGroups, ...
    {
      const int gi = tid / NC, c = tid % NC;
      for (int i = gi; i < n_list; i += kGroups) {
        const int4 w = list[i];
        if (lseg[i] > kShort) continue;
        const ColState st = merge_column<D, GS>(p.records + (size_t)w.x * RS, 0, 1, lseg[i], c);
        store_column(p.out + ((size_t)w.w * p.n_qh + lh0[i]) * D + c * 4, st);
      }
    }
    // long merges: the whole CTA, one item at a time
    for (int i = 0; i < n_list; ++i) {
      const int4 w = list[i];
      const int nseg = lseg[i];
      if (nseg <= kShort) continue;
      const int q = w.y, lg = w.z, v = w.w, h0 = lh0[i];
      // thread (record lane rl, column cc of the chunk) merges records rl,
      // rl + R, ... of column c online (powers of two: shifts and masks only)
      constexpr int kLogNC = __builtin_ctz(NC);
      const int ncq = NC >> lg, R = (kCombineThreads / NC) << lg;
      const int cc = tid & (ncq - 1), rl = tid >> (kLogNC - lg);
      const int c = q * ncq + cc;
      ColState st = merge_column<D, GS>(p.records + (size_t)w.x * RS, rl, R, nseg, c);
      part[tid] = st;
      __syncthreads();
      if (rl == 0) {
        for (int r0 = 1; r0 < R; r0 += 8) {  // the other record lanes' states, eight at a time
          float mm[8], ll[8];
          float4 a[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const bool in = r0 + k < R;
            const ColState o = part[(in ? r0 + k : 0) * ncq + cc];
            mm[k] = in ? o.m : -INFINITY;
            ll[k] = in ? o.l : 0.f;
            a[k] = in ? o.o : make_float4(0.f, 0.f, 0.f, 0.f);
          }
          absorb_batch<8>(st, mm, ll, a);
        }
        store_column(p.out + ((size_t)v * p.n_qh + h0) * D + c * 4, st);
      }
      __syncthreads();
    }
  }
}

template <int D, int GS>
cudaError_t launch_combine_t(const DecodeParams &p, int n_warps, int sms, cudaStream_t stream) {
  const int n_streams = p.n_layers * p.n_seq * p.n_kvh * p.n_sub;
  constexpr int NC = GS * D / 4;
  const long long items = (long long)n_streams * (NC / (16 < NC ? 16 : NC));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(items < 2 * sms ? items : 2 * sms));
  cfg.blockDim = dim3(kCombineThreads);
  cfg.dynamicSmemBytes = (size_t)(p.n_seq + 1) * sizeof(int);  // prefix sums (<= 32.8 KB)
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, combine_kernel<D, GS>, p, n_warps);
}

}  // namespace

cudaError_t launch_combine(const DecodeParams &p, int head_dim, int gs, int n_warps, int sms,
                           cudaStream_t stream) {
  if (p.n_seq <= 0) return cudaSuccess;
  if (head_dim == 64) {
    if (gs == 4) return launch_combine_t<64, 4>(p, n_warps, sms, stream);
    if (gs == 2) return launch_combine_t<64, 2>(p, n_warps, sms, stream);
    return launch_combine_t<64, 1>(p, n_warps, sms, stream);
  }
  if (gs == 4) return launch_combine_t<128, 4>(p, n_warps, sms, stream);
  if (gs == 2) return launch_combine_t<128, 2>(p, n_warps, sms, stream);
  return launch_combine_t<128, 1>(p, n_warps, sms, stream);
}

}  // namespace kvattn
