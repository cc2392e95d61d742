// Combine kernel: log-sum-exp merge of the partial records of split streams
// (third launch of a step for the bf16 cache).
//
// The decode kernel cuts the flattened unit list into equal per-warp shares; a
// stream that crosses share boundaries leaves one record (acc[GS][d] relative
// to 2^m, m[GS], l[GS]; log2 units) per share it touches.  One CTA per stream
// recomputes the same split from the sequence lengths, and for a split stream
// merges its records ("Qwen3-8B inference engine from scratch in C++/CUDA",
// section 4.4.1: blockwise softmax never materialises the full score row; the
// blocks are recombined by rescaling with the running maximum):
//   M = max_r m_r,  L = sum_r 2^(m_r - M) l_r,  out = sum_r 2^(m_r - M) acc_r / L.
// Every thread merges a subset of the records of one float4 column online (a
// running maximum, normaliser and sum, with all its loads issued at once),
// then the record lanes of each column are merged in shared memory: one or
// two L2 round trips per split stream.  The kernel is launched as a
// programmatic dependent of the decode kernel: it plans while the decode grid
// drains and waits for it only before reading records.
#include <mutex>
#include <set>

#include "decode_common.cuh"

namespace kvattn {

namespace {

constexpr int kCombineThreads = 512;

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
__global__ void __launch_bounds__(kCombineThreads)
    combine_kernel(const __grid_constant__ DecodeParams p, int n_warps) {
  constexpr int RS = record_floats(GS, D);
  constexpr int NC = GS * D / 4;             // float4 columns of a record's accumulator
  constexpr int R = kCombineThreads / NC;    // record lanes per column
  constexpr int U = 8;                       // records in flight per thread
  static_assert(kCombineThreads % NC == 0, "columns must tile the CTA");
  extern __shared__ int csmem[];
  int *scratch = csmem;                                         // 32 ints
  ColState *part = reinterpret_cast<ColState *>(csmem + 32);    // [R][NC]
  int *pref = csmem + 32 + (int)(sizeof(ColState) / 4) * kCombineThreads;

  const int tid = threadIdx.x;
  long long T = 0;
  if (!plan_units<kCombineThreads>(p, pref, scratch, T)) return;
  const int spu = p.n_kvh * p.n_sub;
  const int sid = blockIdx.x;
  const int b = sid / spu, si = sid % spu;
  const int units = pref[b + 1] - pref[b];
  if (units == 0) return;
  const long long nwa = min((long long)n_warps, max(1LL, (T + p.min_units - 1) / p.min_units));
  const long long F = (long long)spu * pref[b] + (long long)si * units, E = F + units;
  const long long w0 = owner_of(F, T, nwa), w1 = owner_of(E - 1, T, nwa);
  const int nseg = (int)(w1 - w0 + 1);
  if (nseg <= 1) return;  // written by the decode kernel directly
  const int h0 = (si / p.n_sub) * GS * p.n_sub + (si % p.n_sub) * GS;
  __nv_bfloat16 *outp = p.out + ((size_t)b * p.n_qh + h0) * D;
  const float *r0 = p.records + (size_t)(sid + w0) * RS;

  pdl_wait_primary();  // the decode grid's records are complete and visible

  // thread (record lane rl, column c) merges records rl, rl + R, ... online
  const int c = tid % NC, rl = tid / NC;
  const int hc = (c * 4) / D;
  ColState st = {-INFINITY, 0.f, make_float4(0.f, 0.f, 0.f, 0.f)};
  for (int s0 = rl; s0 < nseg; s0 += R * U) {
    float mm[U], ll[U];
    float4 a[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int s = s0 + u * R;
      if (s < nseg) {
        const float *rs = r0 + (size_t)s * RS;
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
  part[rl * NC + c] = st;
  __syncthreads();
  if (rl == 0) {
    for (int r = 1; r < R; ++r) {
      const ColState q = part[r * NC + c];
      absorb(st, q.m, q.l, q.o);
    }
    const float inv = st.l > 0.f ? 1.f / st.l : 0.f;
    __nv_bfloat162 *dst = reinterpret_cast<__nv_bfloat162 *>(outp + c * 4);
    dst[0] = __floats2bfloat162_rn(st.o.x * inv, st.o.y * inv);
    dst[1] = __floats2bfloat162_rn(st.o.z * inv, st.o.w * inv);
  }
}

template <int D, int GS>
cudaError_t launch_combine_t(const DecodeParams &p, int n_warps, cudaStream_t stream) {
  const int grid = p.n_seq * p.n_kvh * p.n_sub;
  const size_t fixed = 32 * sizeof(int) + sizeof(ColState) * kCombineThreads;
  const size_t smem = fixed + (p.n_seq + 1) * sizeof(int);
  auto kern = combine_kernel<D, GS>;
  static std::mutex mu;
  static std::set<int> configured;  // devices whose shared-memory limit is set
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!configured.count(dev)) {
      err = cudaFuncSetAttribute(
          kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
          (int)(fixed + (KVATTN_MAX_SEQS + 1) * sizeof(int)));
      if (err != cudaSuccess) return err;
      configured.insert(dev);
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kCombineThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p, n_warps);
}

}  // namespace

cudaError_t launch_combine(const DecodeParams &p, int head_dim, int gs, int n_warps,
                           cudaStream_t stream) {
  if (p.n_seq <= 0) return cudaSuccess;
  if (head_dim == 64) {
    if (gs == 4) return launch_combine_t<64, 4>(p, n_warps, stream);
    if (gs == 2) return launch_combine_t<64, 2>(p, n_warps, stream);
    return launch_combine_t<64, 1>(p, n_warps, stream);
  }
  if (gs == 4) return launch_combine_t<128, 4>(p, n_warps, stream);
  if (gs == 2) return launch_combine_t<128, 2>(p, n_warps, stream);
  return launch_combine_t<128, 1>(p, n_warps, stream);
}

}  // namespace kvattn
