// Combine kernel: log-sum-exp merge of the streams the decode kernel's work
// split cut across warp shares (second launch of a step).
//
// A split stream leaves one partial record (acc[GS][d] relative to 2^m,
// m[GS], l[GS]; log2 units) per share it touches, in consecutive slots, and
// its first share writes (first share, shares) into the stream's hand-off
// entry ((0, 0) for a stream one share holds); this kernel merges the records
// ("Qwen3-8B inference engine from scratch in C++/CUDA", section 4.4.1: the
// blockwise softmax recombines its blocks by rescaling with the running
// maximum):
//   M = max_r m_r,  L = sum_r 2^(m_r - M) l_r,  out = sum_r 2^(m_r - M) acc_r / L.
// A stream cut into many shares has its columns split into up to four items,
// so that one round of loads covers its records.  Two CTAs per SM at most;
// CTA c looks at items c, c + gridDim.x, ...: its threads read those items'
// hand-off entries at once and list the merges to do.  Every thread merges a
// subset of the records of one float4 column online (running maximum,
// normaliser and sum, with all its loads issued at once), then the record
// lanes of each column are merged in shared memory.  The
// kernel is launched as a programmatic dependent of the decode kernel and
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

__device__ __forceinline__ void absorb(ColState &st, float m, float l, float4 a) {
  if (m == -INFINITY) return;
  const float mn = fmaxf(st.m, m);
  const float so = (st.m == -INFINITY) ? 0.f : exp2f(st.m - mn);
  const float sa = exp2f(m - mn);
  st.l = st.l * so + l * sa;
  st.o.x = st.o.x * so + a.x * sa;
  st.o.y = st.o.y * so + a.y * sa;
  st.o.z = st.o.z * so + a.z * sa;
  st.o.w = st.o.w * so + a.w * sa;
  st.m = mn;
}

template <int D, int GS>
__global__ void __launch_bounds__(kCombineThreads, 2)
    combine_kernel(const __grid_constant__ DecodeParams p, int n_streams) {
  constexpr int RS = record_floats(GS, D);
  constexpr int NC = GS * D / 4;  // float4 columns of a record's accumulator
  // a long stream's columns may be split into up to kMaxChunks items (of at
  // least 32 columns each) that different CTAs merge
  constexpr int kMaxChunks = NC >= 128 ? 4 : NC >= 64 ? 2 : 1;
  constexpr int U = 16;  // records in flight per thread
  static_assert(kCombineThreads % NC == 0, "columns must tile the CTA");
  __shared__ ColState part[kCombineThreads];  // [record lane][column]
  __shared__ int4 list[kCombineThreads];      // (stream, chunk, chunks, first share)
  __shared__ int lseg[kCombineThreads];
  __shared__ int n_list;

  const int tid = threadIdx.x;
  const int spu = p.n_kvh * p.n_sub;
  pdl_wait_primary();  // the decode grid's records and hand-off entries are visible

  // item i: chunk i / n_streams of stream i % n_streams; CTA c takes items
  // c, c + gridDim.x, ...
  const long long n_items = (long long)n_streams * kMaxChunks;
  const long long stride = (long long)gridDim.x * kCombineThreads;
  for (long long base = blockIdx.x; base < n_items; base += stride) {
    if (tid == 0) n_list = 0;
    __syncthreads();
    const long long it = base + (long long)tid * gridDim.x;
    if (it < n_items) {
      const int sid = (int)(it % n_streams), q = (int)(it / n_streams);
      const int2 m = __ldcg(p.meta + sid);
      const int nseg = m.y;
      // fewest chunks whose record lanes cover the shares in one round
      int nch = 1;
      while (nch < kMaxChunks && nseg > (kCombineThreads * nch / NC) * U) nch *= 2;
      if (nseg > 1 && q < nch) {
        const int k = atomicAdd(&n_list, 1);
        list[k] = make_int4(sid, q, nch, m.x);
        lseg[k] = nseg;
      }
    }
    __syncthreads();
    for (int i = 0; i < n_list; ++i) {
      const int4 w = list[i];
      const int sid = w.x, q = w.y, nch = w.z, w0 = w.w, nseg = lseg[i];
      const int b = sid / spu, si = sid % spu;
      const int h0 = (si / p.n_sub) * GS * p.n_sub + (si % p.n_sub) * GS;
      const float *r0 = p.records + (size_t)(sid + w0) * RS;
      // thread (record lane rl, column cc of the chunk) merges records rl,
      // rl + R, ... of column c online
      const int ncq = NC / nch, R = kCombineThreads / ncq;
      const int cc = tid % ncq, rl = tid / ncq;
      const int c = q * ncq + cc;
      const int hc = (c * 4) / D;
      ColState st = {-INFINITY, 0.f, make_float4(0.f, 0.f, 0.f, 0.f)};
      for (int s0 = rl; s0 < nseg; s0 += R * U) {
        float mm[U], ll[U];
        float4 a[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int r = s0 + u * R;
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
#pragma unroll
        for (int u = 0; u < U; ++u) absorb(st, mm[u], ll[u], a[u]);
      }
      part[tid] = st;
      __syncthreads();
      if (rl == 0) {
        for (int r = 1; r < R; ++r) {
          const ColState o = part[r * ncq + cc];
          absorb(st, o.m, o.l, o.o);
        }
        const float inv = st.l > 0.f ? 1.f / st.l : 0.f;
        __nv_bfloat162 *dst =
            reinterpret_cast<__nv_bfloat162 *>(p.out + ((size_t)b * p.n_qh + h0) * D + c * 4);
        dst[0] = __floats2bfloat162_rn(st.o.x * inv, st.o.y * inv);
        dst[1] = __floats2bfloat162_rn(st.o.z * inv, st.o.w * inv);
      }
      __syncthreads();
    }
  }
}

template <int D, int GS>
cudaError_t launch_combine_t(const DecodeParams &p, int sms, cudaStream_t stream) {
  const int n_streams = p.n_seq * p.n_kvh * p.n_sub;
  cudaLaunchConfig_t cfg = {};
  const long long items = (long long)n_streams * (GS * D / 4 >= 128 ? 4 : GS * D / 4 >= 64 ? 2 : 1);
  cfg.gridDim = dim3((unsigned)(items < 2 * sms ? items : 2 * sms));
  cfg.blockDim = dim3(kCombineThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, combine_kernel<D, GS>, p, n_streams);
}

}  // namespace

cudaError_t launch_combine(const DecodeParams &p, int head_dim, int gs, int sms,
                           cudaStream_t stream) {
  if (p.n_seq <= 0) return cudaSuccess;
  if (head_dim == 64) {
    if (gs == 4) return launch_combine_t<64, 4>(p, sms, stream);
    if (gs == 2) return launch_combine_t<64, 2>(p, sms, stream);
    return launch_combine_t<64, 1>(p, sms, stream);
  }
  if (gs == 4) return launch_combine_t<128, 4>(p, sms, stream);
  if (gs == 2) return launch_combine_t<128, 2>(p, sms, stream);
  return launch_combine_t<128, 1>(p, sms, stream);
}

}  // namespace kvattn
