// RoPE + append kernel: the first of the two launches of one decode step.
//
// One CTA per sequence b:
//  * cos/sin of the new token's position, computed in double from the host's
//    rope_theta^(-2i/d) table and rounded to fp32 ("C17 CPU-first LLM
//    inference engine", section 4.4 "Attention: GQA + RoPE": half-split pairs
//    (i, i + d/2); "LLM inference from smollm3.go", section "Positional
//    encoding": the angle depends on position, head size and theta);
//  * every query head rotated in fp32 and pre-multiplied by scale * log2(e),
//    so the decode kernel's scores come out in log2 units;
//  * the new key rotated with fp32 products and sums each rounded on its own
//    (no fused multiply-add), then stored as bf16 (nearest even) or as int8
//    codes with scale max|x| / 127; the value stored as given or quantised
//    the same way; written to slot L % page of page block_table[b][L / page]
//    ("Qwen3-8B inference engine from scratch in C++/CUDA", section 4.3.1
//    "Paged KV cache"; smollm3.go page, section "int8 weight-only
//    quantization");
//  * the stream arrival counters of the sequence reset to zero for the
//    decode kernel that follows.
// It lets the dependent decode kernel launch early (programmatic dependent
// launch); that kernel waits for this grid before it reads anything written here.
#include "kvattn_internal.cuh"

namespace kvattn {

namespace {

constexpr int kRopeThreads = 128;

__device__ __forceinline__ float bf(const __nv_bfloat16 x) { return __bfloat162float(x); }

// Storage rotation of pair (lo, hi) with fp32 c, s: each product and sum is
// rounded separately (the _rn intrinsics are never fused).
__device__ __forceinline__ void rot_store(float lo, float hi, float c, float s, float &a,
                                          float &b) {
  a = __fsub_rn(__fmul_rn(lo, c), __fmul_rn(hi, s));
  b = __fadd_rn(__fmul_rn(hi, c), __fmul_rn(lo, s));
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
  return v;
}

// Quantise one row of d fp32 values held by one warp (d/32 per lane, element
// lane + 32 * k) to int8 codes and an fp32 scale.
template <int D>
__device__ __forceinline__ void quant_row_warp(const float (&x)[D / 32], int8_t *codes,
                                               float *scale, int lane) {
  float a = 0.f;
#pragma unroll
  for (int k = 0; k < D / 32; ++k) a = fmaxf(a, fabsf(x[k]));
  a = warp_max(a);
  if (a == 0.f) {
#pragma unroll
    for (int k = 0; k < D / 32; ++k) codes[lane + 32 * k] = 0;
    if (lane == 0) *scale = 0.f;
    return;
  }
  const float sc = __fdiv_rn(a, 127.0f);
#pragma unroll
  for (int k = 0; k < D / 32; ++k) {
    float r = rintf(__fdiv_rn(x[k], sc));
    r = fminf(fmaxf(r, -127.f), 127.f);
    codes[lane + 32 * k] = static_cast<int8_t>(static_cast<int>(r));
  }
  if (lane == 0) *scale = sc;
}

template <int D>
__global__ void __launch_bounds__(kRopeThreads) rope_append_kernel(const __grid_constant__ RopeParams p) {
  pdl_launch_dependents();
  constexpr int H = D / 2;
  __shared__ float cs_c[H], cs_s[H];
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  const int L = p.seq_lens[b];
  const int pos = p.positions[b];
  const long long cap = (long long)p.max_pages * p.page_size;
  const bool len_ok = L >= 0 && (long long)L + 1 <= cap;
  int page = -1;
  if (len_ok) page = p.block_table[(size_t)b * p.max_pages + L / p.page_size];
  const bool page_ok = len_ok && page >= 0 && page < p.num_pages;
  if (tid == 0) {
    if (!len_ok) atomicOr(p.status, KVATTN_DEV_BAD_LEN);
    else if (!page_ok) atomicOr(p.status, KVATTN_DEV_BAD_PAGE);
  }
  for (int s = tid; s < p.streams_per_seq; s += kRopeThreads)
    p.counters[(size_t)b * p.streams_per_seq + s] = 0u;

  for (int i = tid; i < H; i += kRopeThreads) {
    float c = 1.f, s = 0.f;
    if (p.use_rope) {
      double sd, cd;
      sincos((double)pos * p.inv_freq[i], &sd, &cd);
      c = (float)cd;
      s = (float)sd;
    }
    cs_c[i] = c;
    cs_s[i] = s;
  }
  __syncthreads();

  // queries: rotated in fp32, pre-scaled
  const __nv_bfloat16 *qb = p.q + (size_t)b * p.n_qh * D;
  float *qo = p.qhat + (size_t)b * p.n_qh * D;
  for (int idx = tid; idx < p.n_qh * H; idx += kRopeThreads) {
    const int h = idx / H, i = idx % H;
    const float lo = bf(qb[h * D + i]), hi = bf(qb[h * D + i + H]);
    float a = lo, c2 = hi;
    if (p.use_rope) rot_store(lo, hi, cs_c[i], cs_s[i], a, c2);
    qo[h * D + i] = a * p.qscale;
    qo[h * D + i + H] = c2 * p.qscale;
  }
  if (!page_ok) return;

  const int off = L % p.page_size;
  const size_t slot0 = ((size_t)page * p.n_kvh) * p.page_size + off;  // head 0
  const __nv_bfloat16 *kb = p.k_new + (size_t)b * p.n_kvh * D;
  const __nv_bfloat16 *vb = p.v_new + (size_t)b * p.n_kvh * D;
  if (!p.kv_int8) {
    __nv_bfloat16 *kp = static_cast<__nv_bfloat16 *>(p.k_pages);
    __nv_bfloat16 *vp = static_cast<__nv_bfloat16 *>(p.v_pages);
    for (int idx = tid; idx < p.n_kvh * H; idx += kRopeThreads) {
      const int j = idx / H, i = idx % H;
      const size_t row = (slot0 + (size_t)j * p.page_size) * D;
      const float lo = bf(kb[j * D + i]), hi = bf(kb[j * D + i + H]);
      float a = lo, c2 = hi;
      if (p.use_rope) rot_store(lo, hi, cs_c[i], cs_s[i], a, c2);
      kp[row + i] = __float2bfloat16_rn(a);
      kp[row + i + H] = __float2bfloat16_rn(c2);
      vp[row + i] = vb[j * D + i];
      vp[row + i + H] = vb[j * D + i + H];
    }
    return;
  }
  // int8: one warp per KV head row; element e = lane + 32k
  int8_t *kp = static_cast<int8_t *>(p.k_pages);
  int8_t *vp = static_cast<int8_t *>(p.v_pages);
  const int warp = tid / 32, lane = tid % 32;
  for (int j = warp; j < p.n_kvh; j += kRopeThreads / 32) {
    const size_t srow = slot0 + (size_t)j * p.page_size;
    float xk[D / 32], xv[D / 32];
#pragma unroll
    for (int k = 0; k < D / 32; ++k) {
      const int e = lane + 32 * k;
      const int i = e % H;
      const float lo = bf(kb[j * D + i]), hi = bf(kb[j * D + i + H]);
      float a = lo, c2 = hi;
      if (p.use_rope) rot_store(lo, hi, cs_c[i], cs_s[i], a, c2);
      xk[k] = (e < H) ? a : c2;
      xv[k] = bf(vb[j * D + e]);
    }
    quant_row_warp<D>(xk, kp + srow * D, p.k_scales + srow, lane);
    quant_row_warp<D>(xv, vp + srow * D, p.v_scales + srow, lane);
  }
}

}  // namespace

cudaError_t launch_rope_append(const RopeParams &p, cudaStream_t stream) {
  if (p.n_seq <= 0) return cudaSuccess;
  if (p.head_dim == 64)
    rope_append_kernel<64><<<p.n_seq, kRopeThreads, 0, stream>>>(p);
  else
    rope_append_kernel<128><<<p.n_seq, kRopeThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace kvattn
