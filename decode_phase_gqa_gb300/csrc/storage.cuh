// Storage recipe of the slot a decode step appends: the new key rotated and
// rounded exactly as the cache stores it, and the int8 quantisation of a row.
//
//  * cos/sin of the new token's position: the angle position * theta^(-2i/d)
//    in double (host frequency table), cos/sin of that double, rounded to
//    fp32 ("C17 CPU-first LLM inference engine", section 4.4 "Attention: GQA +
//    RoPE": half-split pairs (i, i + d/2));
//  * the key rotated with fp32 products and sums each rounded on its own (no
//    fused multiply-add), stored as bf16 (nearest even) or as int8 codes with
//    scale max|x| / 127 ("LLM inference from smollm3.go", section "int8
//    weight-only quantization"); the value stored as given or quantised the
//    same way.
// These bytes are the only ones of the pool a step writes, and they must match
// the recipe bit for bit, hence the correctly rounded cos/sin.
//
// A warp holds one row of d values: lane l owns the rotation pairs (i, i + d/2)
// for i = l + 32k, k < d/64, as x[k] = row[i] and x[d/64 + k] = row[i + d/2].
#pragma once

#include "kvattn_internal.cuh"

namespace kvattn {

#include "angle_table.inc"  // kSinCosStep[j]: sin, cos of j pi / 256 (float-float)

// Element index of slot k of a lane's row share (see above).
template <int D>
__device__ __forceinline__ int row_elem(int lane, int k) {
  return k < D / 64 ? lane + 32 * k : D / 2 + lane + 32 * (k - D / 64);
}

// Rotation of pair (lo, hi) by fp32 (c, s) with every product and sum rounded
// on its own (the _rn intrinsics are never fused).
__device__ __forceinline__ void rot_store(float lo, float hi, float c, float s, float &a,
                                          float &b) {
  a = __fsub_rn(__fmul_rn(lo, c), __fmul_rn(hi, s));
  b = __fadd_rn(__fmul_rn(hi, c), __fmul_rn(lo, s));
}

// ---- fp32 cos/sin of the double angle pos * inv_freq, correctly rounded ----
// The recipe is fl32(cos(phi)), fl32(sin(phi)) of the double phi = fl64(pos *
// inv_freq).  Double-precision sine/cosine run on the slow FP64 pipe, so the
// values are formed in float-float arithmetic (an unevaluated sum hi + lo of
// two floats, about 48 bits) and rounded to fp32; only a value that lands
// within kAngleEps of an fp32 rounding midpoint, where the float-float error
// could decide the rounding, is recomputed with double sincos.
//  1. Cody-Waite reduction in double: k = an integer near phi * 2/pi (from
//     fp32), r = phi - k * pio2_hi - k * pio2_lo with pio2_hi = fl64(pi/2) and
//     pio2_lo = fl64(pi/2 - pio2_hi); the first step is exact (the difference
//     is a multiple of ulp(pio2_hi) below 1 in magnitude), so |r| <= 0.87 with
//     an error near 2^-53.
//  2. r split into a float head rh (its top 24 bits) and tail rl.
//  3. A second reduction by j steps of pi/256 (j = nearest integer to
//     rh * 256/pi, |j| <= 72): r' = r - j pi/256 as float-float (the step is
//     split into a 17-bit head, so j * head is exact, and two tails), |r'| <=
//     0.0062.
//  4. sin(r') = r' + ds, cos(r') = 1 + dc with dc = -t/2 + t^2/24 (t = r'^2 as
//     float-float) and ds = r' t (-1/6 + t/120) in fp32: the dropped terms are
//     below 2^-60.
//  5. sin(r) = S + S dc + C r' + C ds, cos(r) = C + C dc - S r' - S ds with
//     (S, C) = (sin, cos)(j pi/256) from a float-float table, then the
//     quadrant k mod 4.
// The float-float result is within 2^-46 of the exact value (4 FP64
// operations and about 100 fp32 operations per angle).
struct FF {
  float hi, lo;
};

__device__ __forceinline__ FF ff_fast2(float a, float b) {  // |a| >= |b|
  const float s = __fadd_rn(a, b);
  return {s, __fsub_rn(b, __fsub_rn(s, a))};
}
__device__ __forceinline__ FF ff_two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  return {s, __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb))};
}
__device__ __forceinline__ FF ff_two_prod(float a, float b) {
  const float p = __fmul_rn(a, b);
  return {p, __fmaf_rn(a, b, -p)};
}
__device__ __forceinline__ FF ff_mul(FF x, FF y) {
  const float p = __fmul_rn(x.hi, y.hi);
  float e = __fmaf_rn(x.hi, y.hi, -p);
  e = __fmaf_rn(x.hi, y.lo, e);
  e = __fmaf_rn(x.lo, y.hi, e);
  return ff_fast2(p, e);
}
__device__ __forceinline__ FF ff_add(FF x, FF y) {
  const FF s = ff_two_sum(x.hi, y.hi);
  return ff_fast2(s.hi, __fadd_rn(__fadd_rn(s.lo, x.lo), y.lo));
}
__device__ __forceinline__ FF ff_add(FF x, float y) {
  const FF s = ff_two_sum(x.hi, y);
  return ff_fast2(s.hi, __fadd_rn(s.lo, x.lo));
}
__device__ __forceinline__ FF ff_neg(FF x) { return {-x.hi, -x.lo}; }

constexpr double kPio2Hi = 0x1.921fb54442d18p+0;   // fl64(pi/2)
constexpr double kPio2Lo = 0x1.1a62633145c07p-54;  // fl64(pi/2 - kPio2Hi)
constexpr float kStepHi = 0x1.921fp-7f;            // pi/256 to 17 bits
constexpr float kStepLo = 0x1.6a8886p-24f;         // fl32(pi/256 - kStepHi)
constexpr float kStepLo2 = -0x1.73dcb4p-50f;       // the rest
constexpr float kAngleEps = 0x1p-44f;

// true when rounding hi + lo to fp32 could depend on an error of kAngleEps
__device__ __forceinline__ bool near_midpoint(FF v) {
  const float f = __fadd_rn(v.hi, v.lo);
  if (f != v.hi || f == 0.f) return true;
  const int b = __float_as_int(f);
  // neighbour on the side of lo (integer order of the bits is magnitude order)
  const bool away = (v.lo > 0.f) == (f > 0.f);
  const float half_gap = 0.5f * fabsf(__int_as_float(away ? b + 1 : b - 1) - f);
  return fabsf(half_gap - fabsf(v.lo)) <= kAngleEps;
}

// The rare slow path of store_angle below: cos/sin in double, then rounded.
// Kept out of line, so that the kernels carry one copy of it.
static __device__ __noinline__ void angle_slow(double phi, float &c, float &s) {
  double sd, cd;
  sincos(phi, &sd, &cd);
  c = (float)cd;
  s = (float)sd;
}

// fp32 cos/sin of the double angle pos * inv_freq, as (float)cos / (float)sin
// of that double would round them.  `table` is a copy of kSinCosStep (in
// shared memory: a lane-divergent read of global memory would queue behind
// the SM's tile copies).
__device__ __forceinline__ void store_angle_inl(int pos, double inv_freq, const float4 *table, float &c,
                                               float &s) {
  const double phi = (double)pos * inv_freq;
  // the quadrant from an fp32 estimate of phi (its error and that of the
  // product with 2/pi stay below 5 * 2^-24 phi): while phi < 2^18 the
  // integer k is within 0.55 of phi * 2/pi, so |r| <= 0.87
  const float phf = __fmul_rn((float)pos, (float)inv_freq);
  bool slow = !(phf < 0x1p18f);
  if (pos == 0 || inv_freq == 0.0) {
    c = 1.f;
    s = 0.f;
    return;
  }
  if (!slow) {
    // 1. quadrant and reduced angle
    const int k = __float2int_rn(__fmul_rn(phf, 0x1.45f306p-1f));  // phi * 2/pi
    const int q = k & 3;
    const double kd = (double)k;
    const double r = __fma_rn(-kd, kPio2Lo, __fma_rn(-kd, kPio2Hi, phi));
    // 2. rh = r with its 29 low mantissa bits cleared, rl = the rest
    const unsigned long long rb = (unsigned long long)__double_as_longlong(r);
    const int e = (int)((rb >> 52) & 0x7ff) - 1023;
    const unsigned sign = (unsigned)(rb >> 63) << 31;
    float rh = 0.f, rl = 0.f;  // |r| < 2^-126 only when phi == 0 (handled above)
    if (e >= -126)
      rh = __uint_as_float(sign | ((unsigned)(e + 127) << 23) | (unsigned)((rb >> 29) & 0x7fffff));
    if (e >= -74) {  // the tail's scale 2^(e - 52) is a normal float
      const float tail = __uint2float_rn((unsigned)(rb & 0x1fffffff));  // 29-bit integer
      rl = __fmul_rn(tail, __uint_as_float((unsigned)(e - 52 + 127) << 23));
      if (sign) rl = -rl;
    }
    // 3. r' = r - j pi/256
    const int j = __float2int_rn(__fmul_rn(rh, 0x1.45f306p+6f));  // rh * 256/pi
    const int aj = abs(j);
    if (aj <= 72) {
      const float jf = (float)j;
      FF rp = ff_add(FF{__fsub_rn(rh, __fmul_rn(jf, kStepHi)), 0.f}, rl);  // (exact difference)
      rp = ff_add(rp, ff_two_prod(-jf, kStepLo));
      rp = ff_add(rp, __fmul_rn(-jf, kStepLo2));
      // 4. dc, ds
      const float th = __fmul_rn(rp.hi, rp.hi);
      const FF t = ff_fast2(th, __fmaf_rn(2.f * rp.hi, rp.lo, __fmaf_rn(rp.hi, rp.hi, -th)));
      const FF dc =
          ff_add(FF{-0.5f * t.hi, -0.5f * t.lo}, __fmul_rn(__fmul_rn(t.hi, t.hi), 1.f / 24.f));
      const float ds = __fmul_rn(__fmul_rn(rp.hi, t.hi), __fmaf_rn(t.hi, 1.f / 120.f, -1.f / 6.f));
      // 5. recombination with the table
      const float4 tb = table[aj];
      const FF S = j < 0 ? FF{-tb.x, -tb.y} : FF{tb.x, tb.y};
      const FF C = {tb.z, tb.w};
      const FF s1 = ff_add(ff_add(S, ff_mul(S, dc)), ff_add(ff_mul(C, rp), __fmul_rn(C.hi, ds)));
      const FF c1 =
          ff_add(ff_add(C, ff_mul(C, dc)), ff_add(ff_mul(ff_neg(S), rp), -__fmul_rn(S.hi, ds)));
      const FF sv = (q == 0) ? s1 : (q == 1) ? c1 : (q == 2) ? ff_neg(s1) : ff_neg(c1);
      const FF cv = (q == 0) ? c1 : (q == 1) ? ff_neg(s1) : (q == 2) ? ff_neg(c1) : s1;
      slow = near_midpoint(sv) || near_midpoint(cv);
      s = sv.hi;
      c = cv.hi;
    } else {
      slow = true;
    }
  }
  if (slow) angle_slow(phi, c, s);
}

// The same out of line, so that the decode kernels carry one copy of it
// (their latency-bound phases stalled on instruction fetch with more code);
// the prefill append kernel, a short kernel run by many CTAs, inlines it.
static __device__ __noinline__ void store_angle(int pos, double inv_freq, const float4 *table, float &c,
                                            float &s) {
  store_angle_inl(pos, inv_freq, table, c, s);
}

// Quantise one warp-held row of d fp32 values: int8 codes (lane's slots, in
// the order of x) and the row's fp32 scale (0 for an all-zero row, whose codes
// are 0).
template <int D>
__device__ __forceinline__ float quant_row_warp(const float (&x)[D / 32], int8_t (&codes)[D / 32]) {
  float a = 0.f;
#pragma unroll
  for (int k = 0; k < D / 32; ++k) a = fmaxf(a, fabsf(x[k]));
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, m));
  if (a == 0.f) {
#pragma unroll
    for (int k = 0; k < D / 32; ++k) codes[k] = 0;
    return 0.f;
  }
  const float sc = __fdiv_rn(a, 127.0f);
#pragma unroll
  for (int k = 0; k < D / 32; ++k) {
    float r = rintf(__fdiv_rn(x[k], sc));
    r = fminf(fmaxf(r, -127.f), 127.f);
    codes[k] = static_cast<int8_t>(static_cast<int>(r));
  }
  return sc;
}

// Bytes of a warp's buffer for the new token's row: first the raw key and
// value rows (bf16, d elements each), then in their place the stored form
// (key row, value row, int8: the two scales).
template <int D, bool INT8>
__host__ __device__ constexpr int new_row_bytes() {
  return 4 * D;
}

// Form the stored key and value of the new token for one (sequence, KV head)
// from the raw rows (bf16 key row then value row) that `buf` holds, at RoPE
// position pos, into `buf` (natural element order; int8: the two scales
// follow the rows).  Ends with __syncwarp().
template <int D, bool INT8>
__device__ __forceinline__ void stage_new_row(int pos, const double *inv_freq, const float4 *table,
                                              bool use_rope, int lane, uint8_t *buf) {
  constexpr int PPL = D / 64;
  static_assert(2 * D * (INT8 ? 1 : 2) + (INT8 ? 8 : 0) <= 4 * D, "the stored form fits");
  float xk[D / 32], xv[D / 32];
  const __nv_bfloat16 *raw = reinterpret_cast<const __nv_bfloat16 *>(buf);
#pragma unroll
  for (int k = 0; k < D / 32; ++k) {
    xk[k] = __bfloat162float(raw[row_elem<D>(lane, k)]);
    xv[k] = __bfloat162float(raw[D + row_elem<D>(lane, k)]);
  }
  __syncwarp();  // every lane has read the raw rows before the buffer is rewritten
  if (use_rope) {
    float c[PPL], s[PPL];
#pragma unroll
    for (int k = 0; k < PPL; ++k) store_angle(pos, inv_freq[lane + 32 * k], table, c[k], s[k]);
#pragma unroll
    for (int k = 0; k < PPL; ++k) rot_store(xk[k], xk[PPL + k], c[k], s[k], xk[k], xk[PPL + k]);
  }
  if constexpr (INT8) {
    int8_t kc[D / 32], vc[D / 32];
    const float ks = quant_row_warp<D>(xk, kc);
    const float vs = quant_row_warp<D>(xv, vc);
    int8_t *kr = reinterpret_cast<int8_t *>(buf), *vr = kr + D;
#pragma unroll
    for (int k = 0; k < D / 32; ++k) {
      kr[row_elem<D>(lane, k)] = kc[k];
      vr[row_elem<D>(lane, k)] = vc[k];
    }
    if (lane == 0) {
      float *sc = reinterpret_cast<float *>(buf + 2 * D);
      sc[0] = ks;
      sc[1] = vs;
    }
  } else {
    __nv_bfloat16 *kr = reinterpret_cast<__nv_bfloat16 *>(buf), *vr = kr + D;
#pragma unroll
    for (int k = 0; k < D / 32; ++k) {
      kr[row_elem<D>(lane, k)] = __float2bfloat16_rn(xk[k]);
      vr[row_elem<D>(lane, k)] = __float2bfloat16_rn(xv[k]);
    }
  }
  __syncwarp();
}

// The staged row -> row `row` of a unit's K and V tiles in shared memory
// (16-byte chunk ch of a row at chunk_off(row, ch)) and of its int8 row
// scales sc (K at sc[row], V at sc[16 + row]), and, when slot >= 0, to pool
// row `slot` (the append): one 16-byte chunk per lane.
template <int D, bool INT8, class ChunkOff>
__device__ __forceinline__ void put_new_row(const uint8_t *buf, uint8_t *Ks, uint8_t *Vs, float *sc,
                                            int row, long long slot, void *k_pages, void *v_pages,
                                            float *k_scales, float *v_scales, int lane,
                                            ChunkOff chunk_off) {
  constexpr int RB = D * (INT8 ? 1 : 2);  // bytes of a row
  constexpr int CH = RB / 16;
  static_assert(2 * CH <= 32, "a warp moves the two rows in one pass");
  if (lane < 2 * CH) {
    const bool v = lane >= CH;
    const int c = v ? lane - CH : lane;
    const uint4 x = *reinterpret_cast<const uint4 *>(buf + (v ? RB : 0) + 16 * c);
    *reinterpret_cast<uint4 *>((v ? Vs : Ks) + chunk_off(row, c)) = x;
    if (slot >= 0)
      *reinterpret_cast<uint4 *>(static_cast<uint8_t *>(v ? v_pages : k_pages) + slot * RB +
                                 16 * c) = x;
  }
  if constexpr (INT8) {
    if (lane == 0) {
      const float *s = reinterpret_cast<const float *>(buf + 2 * RB);
      sc[row] = s[0];
      sc[kUnitRows + row] = s[1];
      if (slot >= 0) {
        k_scales[slot] = s[0];
        v_scales[slot] = s[1];
      }
    }
  }
}

}  // namespace kvattn
