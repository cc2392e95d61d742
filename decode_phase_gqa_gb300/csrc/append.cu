// Append kernel: the first of the two launches of one decode step.
//
// One CTA per sequence b writes the new key and value into slot L % page of
// page block_table[b][L / page] (L = seq_lens[b]; "Qwen3-8B inference engine
// from scratch in C++/CUDA", section 4.3.1 "Paged KV cache"):
//  * cos/sin of the new token's position: the angle position * theta^(-2i/d)
//    in double (host frequency table), cos/sin in double, rounded to fp32
//    ("C17 CPU-first LLM inference engine", section 4.4 "Attention: GQA +
//    RoPE": half-split pairs (i, i + d/2));
//  * the key rotated with fp32 products and sums each rounded on its own (no
//    fused multiply-add), stored as bf16 (nearest even) or as int8 codes with
//    scale max|x| / 127 ("LLM inference from smollm3.go", section "int8
//    weight-only quantization"); the value stored as given or quantised the
//    same way.
// These bytes are the only ones of the pool a step writes, and they must match
// the storage recipe bit for bit, hence the double-precision angle.
// The decode kernel is launched as a programmatic dependent of this grid and
// waits for it only before it loads a unit that holds a new token.
#include "kvattn_internal.cuh"

namespace kvattn {

namespace {

constexpr int kAppendThreads = 128;

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

// Quantise one row of d fp32 values held by one warp to int8 codes and an
// fp32 scale.  Lane l holds x[k] = row[l + 32k] for k < d/64 and
// x[d/64 + k] = row[d/2 + l + 32k].
template <int D>
__device__ __forceinline__ void quant_row_warp(const float (&x)[D / 32], int8_t *codes,
                                               float *scale, int lane) {
  constexpr int PPL = D / 64;
  auto index = [&](int k) { return k < PPL ? lane + 32 * k : D / 2 + lane + 32 * (k - PPL); };
  float a = 0.f;
#pragma unroll
  for (int k = 0; k < D / 32; ++k) a = fmaxf(a, fabsf(x[k]));
  a = warp_max(a);
  if (a == 0.f) {
#pragma unroll
    for (int k = 0; k < D / 32; ++k) codes[index(k)] = 0;
    if (lane == 0) *scale = 0.f;
    return;
  }
  const float sc = __fdiv_rn(a, 127.0f);
#pragma unroll
  for (int k = 0; k < D / 32; ++k) {
    float r = rintf(__fdiv_rn(x[k], sc));
    r = fminf(fmaxf(r, -127.f), 127.f);
    codes[index(k)] = static_cast<int8_t>(static_cast<int>(r));
  }
  if (lane == 0) *scale = sc;
}

// Warp w handles KV heads w, w + 4, ...; lane l owns the rotation pairs
// (i, i + d/2) for i = l + 32k.
template <int D>
__global__ void __launch_bounds__(kAppendThreads) append_kernel(const __grid_constant__ AppendParams p) {
  pdl_launch_dependents();
  constexpr int H = D / 2;
  constexpr int PPL = H / 32;  // rotation pairs per lane
  __shared__ float cs_c[H], cs_s[H];
  const int b = blockIdx.x;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int L = __ldg(p.seq_lens + b);
  const int pos = __ldg(p.positions + b);
  const long long cap = (long long)p.max_pages * p.page_size;
  const bool len_ok = L >= 0 && (long long)L + 1 <= cap;
  const int page = len_ok ? __ldg(p.block_table + (size_t)b * p.max_pages + L / p.page_size) : -1;
  const bool page_ok = len_ok && page >= 0 && page < p.num_pages;
  if (tid == 0) {
    if (!len_ok) atomicOr(p.status, KVATTN_DEV_BAD_LEN);
    else if (!page_ok) atomicOr(p.status, KVATTN_DEV_BAD_PAGE);
  }
  if (!page_ok) return;
  for (int i = tid; i < H; i += kAppendThreads) {
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
  for (int j = warp; j < p.n_kvh; j += kAppendThreads / 32) {
    const __nv_bfloat16 *ks = p.k_new + ((size_t)b * p.n_kvh + j) * D;
    const __nv_bfloat16 *vs = p.v_new + ((size_t)b * p.n_kvh + j) * D;
    float rlo[PPL], rhi[PPL], vlo[PPL], vhi[PPL];
#pragma unroll
    for (int k = 0; k < PPL; ++k) {
      const float lo = bf(ks[lane + 32 * k]), hi = bf(ks[lane + 32 * k + H]);
      vlo[k] = bf(vs[lane + 32 * k]);
      vhi[k] = bf(vs[lane + 32 * k + H]);
      rlo[k] = lo;
      rhi[k] = hi;
      if (p.use_rope) rot_store(lo, hi, cs_c[lane + 32 * k], cs_s[lane + 32 * k], rlo[k], rhi[k]);
    }
    const size_t srow = ((size_t)page * p.n_kvh + j) * p.page_size + L % p.page_size;
    if (!p.kv_int8) {
      __nv_bfloat16 *kp = static_cast<__nv_bfloat16 *>(p.k_pages) + srow * D;
      __nv_bfloat16 *vp = static_cast<__nv_bfloat16 *>(p.v_pages) + srow * D;
#pragma unroll
      for (int k = 0; k < PPL; ++k) {
        kp[lane + 32 * k] = __float2bfloat16_rn(rlo[k]);
        kp[lane + 32 * k + H] = __float2bfloat16_rn(rhi[k]);
        vp[lane + 32 * k] = __float2bfloat16_rn(vlo[k]);
        vp[lane + 32 * k + H] = __float2bfloat16_rn(vhi[k]);
      }
    } else {
      float xk[D / 32], xv[D / 32];
#pragma unroll
      for (int k = 0; k < PPL; ++k) {
        xk[k] = rlo[k];
        xk[PPL + k] = rhi[k];
        xv[k] = vlo[k];
        xv[PPL + k] = vhi[k];
      }
      quant_row_warp<D>(xk, static_cast<int8_t *>(p.k_pages) + srow * D, p.k_scales + srow, lane);
      quant_row_warp<D>(xv, static_cast<int8_t *>(p.v_pages) + srow * D, p.v_scales + srow, lane);
    }
  }
}

}  // namespace

cudaError_t launch_append(const AppendParams &p, cudaStream_t stream) {
  if (p.n_seq <= 0) return cudaSuccess;
  if (p.head_dim == 64)
    append_kernel<64><<<p.n_seq, kAppendThreads, 0, stream>>>(p);
  else
    append_kernel<128><<<p.n_seq, kAppendThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace kvattn
