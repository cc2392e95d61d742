// Split-KV flash-decoding kernel, tensor-core inner loop, for the bf16 and the
// int8 KV cache.
//
// Work split.  Every (sequence, KV head, query-head group) is a stream of
// 16-token units; the streams are laid end to end and the flattened unit list
// is cut into equal contiguous shares, one per WARP of the grid.  Warps are
// independent after the CTA's prologue (the per-sequence prefix sums): each
// streams its share through its own ring of shared-memory stages filled by TMA
// tensor copies (cp.async.bulk.tensor.2d, [16 rows][128 or 64 bytes] boxes,
// 128- or 64-byte swizzle so the ldmatrix reads below hit all 32 banks; the
// int8 cache's per-row scales come with the same barrier by cp.async.bulk),
// keeps its softmax state in registers, and at each stream boundary either
// writes the output (a stream inside its share) or a partial record that the
// combine kernel (combine.cu, launched as this grid's programmatic dependent)
// merges.
//
// Per unit the warp computes, with m16n8k16 MMAs (fp32 accumulate):
//   S^T[16 tokens][8] = K[16][d] * Qc^T[d][8]
//   O^T[d][8]        += V^T[d][16] * P^T[16][8]
// The 8 MMA columns carry, for the GS query heads of the group, the head of
// each value and its remainder (x = hi + lo) in the MMA's input type, so
// neither the query nor the softmax weights lose precision to rounding:
// columns h and GS + h are added back together.  K and V are exact in that
// type: bf16 values of the bf16 cache, and int8 codes of the int8 cache
// converted to f16 in registers (every integer below 2^11 is an f16).
// Tokens are the MMA rows, so one K/V block serves every head of the group
// ("Qwen3-8B inference engine from scratch in C++/CUDA", section 4.4.2:
// read the group's KV once for all its query heads), and the online softmax
// ("LLM inference from smollm3.go", section "Self-attention") runs on the
// accumulator fragments in fp32, in log2 units.
//
// Int8 cache (per-row scales ks_t, vs_t, row = scale * codes: "lightLLM, a
// pure-Python inference framework", section 1 "Overview", Int8KV; the dot
// product of the codes times the row scale as in "LLM inference from
// smollm3.go", section "int8 weight-only quantization"):
//   * score_t = (q . codes_t) * ks_t: the query columns are f16 head and
//     remainder of q * 2^kq, kq a power-of-two range scale per stream, and the
//     raw dot product is multiplied by ks_t * 2^-kq;
//   * the value weights p_t vs_t are formed as 2^(s_t - m + log2 vs_t - dmo)
//     with their own running maximum m + dmo, so the largest weight of the
//     stream so far is 1 (no f16 overflow or underflow whatever the scales);
//     dmo is kept relative to m so that log2 vs_t is added to a number near
//     zero (added to a score of 5e5 fp32 would keep it to 1/32 only); the
//     normaliser l keeps the plain softmax maximum m, and the accumulator is
//     brought from 2^(m + dmo) to 2^m when the stream's part ends.
#pragma once

#include <cuda_fp16.h>

#include <map>
#include <mutex>
#include <set>
#include <utility>

#include "decode_common.cuh"
#include "storage.cuh"

namespace kvattn {

template <int D, int GS, bool INT8>
struct MmaCfg {
  static constexpr int W = kDecodeWarps;
  static constexpr int kRowBytes = INT8 ? D : 2 * D;               // one cached row
  static constexpr int kBoxW = kRowBytes < 128 ? kRowBytes : 128;  // bytes per box row
  static constexpr int kChunks = kBoxW / 16;     // 16-byte chunks per box row
  static constexpr int kRegions = kRowBytes / kBoxW;  // boxes per 16-row tile
  static constexpr int kBox = kUnitRows * kBoxW;
  static constexpr int kTile = kRegions * kBox;
  static constexpr int kStage = 2 * kTile;  // K then V
  static constexpr int kScales = INT8 ? 2 * kUnitRows * 4 : 0;  // K then V row scales
  static constexpr int kQBytes = GS * D * 2;  // one stream's raw query rows (bf16)
  static constexpr int kNewBytes = new_row_bytes<D, INT8>();  // the new token's stored row
  // stages per warp: as many as fit a 75 KB CTA (3 CTAs per SM) next to the
  // frequency and angle tables, per-warp query and new-row buffers, barriers and stage
  // pages, the 1 KB alignment slack and 1600 bytes for the per-sequence
  // arrays (batches of up to 132 sequences keep 3 CTAs per SM)
  static constexpr int kTabBytes = (int)sizeof(kSinCosStep);  // sin/cos steps of the angle routine
  static constexpr int kOther = 1024 + 64 + kTabBytes + W * (kQBytes + kNewBytes) + 1024;
  static constexpr int kPerStage = kStage + kScales + 8 + 4;
  static constexpr int kSWFit = (kCtaSmemBudget - kOther - 1600) / (W * kPerStage);
  static constexpr int kSW = kSWFit > 8 ? 8 : kSWFit;
  static constexpr int kKSteps = D / 16;       // MMA k-steps (QK) and m-tiles (PV)
  static constexpr int kLdm = kRowBytes / 32;  // ldmatrix.x4 per tile (2 chunks each)
  static constexpr int kStagesBytes = W * kSW * kStage;
  static constexpr int kScaleOff = kStagesBytes;                  // [W][kSW][32] fp32
  static constexpr int kBarOff = kScaleOff + W * kSW * kScales;
  static constexpr int kFreqOff = kBarOff + W * kSW * 8;  // rope turns per position, float2[D/2]
  static constexpr int kInvOff = kFreqOff + 512;   // rope_theta^(-2i/d), double[D/2]
  // 4 ints of scratch; test builds' never-completed barrier at +16; the warps'
  // new-row barriers (uint64[W]) at +32
  static constexpr int kMiscOff = kInvOff + 512;
  static constexpr int kQOff = kMiscOff + 64;             // [W][GS][D] bf16
  static constexpr int kNewOff = kQOff + W * kQBytes;     // [W][kNewBytes]
  static constexpr int kValidOff = kNewOff + W * kNewBytes;  // [W][kSW] int: page of a stage
  static constexpr int kTabOff = kValidOff + W * kSW * 4;  // copy of kSinCosStep (float4)
  static constexpr int kPrefOff = kTabOff + kTabBytes;
  // fixed part + alignment slack; the per-sequence arrays (prefix sums,
  // lengths, positions: 3 n_seq + 1 ints) follow
  static constexpr int kFixedSmem = kPrefOff + 1024;
  static constexpr int RS = record_floats(GS, D);
  static_assert(kStage % 1024 == 0, "swizzled boxes need 1024-byte alignment");
  static_assert(kSW >= 2, "need at least double buffering");
  static_assert(kQBytes % 16 == 0, "query rows are copied in 16-byte chunks");
  static_assert(kFreqOff % 16 == 0, "turns are read as float2");
  static_assert(kTabOff % 16 == 0 && kTabBytes % 16 == 0, "the angle table is read as float4");
  static_assert(32 + 8 * W <= 64, "the misc area holds the new-row barriers");
  static_assert(kNewOff % 16 == 0 && kNewBytes % 16 == 0, "new rows move in 16-byte chunks");
};

// Byte offset of 16-byte chunk `ch` of row `row` in a [16][kRowBytes] tile
// written by the TMA as kRegions boxes of [16][kBoxW] bytes: within a box the
// chunk index is XORed with row mod 8 (128-byte swizzle: address bits 4-6
// with bits 7-9) or with (row / 2) mod 4 (64-byte swizzle: bits 4-5 with
// bits 7-8).
template <class C>
__device__ __forceinline__ uint32_t tile_off(int row, int ch) {
  const int region = ch / C::kChunks, c = ch % C::kChunks;
  if constexpr (C::kBoxW == 128)
    return (uint32_t)(region * C::kBox + row * 128 + ((c ^ (row & 7)) << 4));
  else
    return (uint32_t)(region * C::kBox + row * 64 + ((c ^ ((row >> 1) & 3)) << 4));
}

__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t u) {
  return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ float f16_round(float x) { return __half2float(__float2half_rn(x)); }
__device__ __forceinline__ float bf16_round(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}

// D (16x8 fp32) += A (16x16 f16, row) * B (16x8 f16, col)
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// 2^k for an integer k in [-126, 127]
__device__ __forceinline__ float pow2i(int k) { return __uint_as_float((uint32_t)(k + 127) << 23); }

// RoPE of the query, fp32 only (the query needs fp32 accuracy): lane l holds
// cos/sin of angles l + 32k of position `pos`, from frac_turns and sincospif.
template <int D>
__device__ __forceinline__ void warp_query_angles(const float2 *turns, int pos, bool rope,
                                                  int lane, float (&cr)[D / 64],
                                                  float (&sr)[D / 64]) {
#pragma unroll
  for (int k = 0; k < D / 64; ++k) {
    cr[k] = 1.f;
    sr[k] = 0.f;
    if (rope) sincospif(2.f * frac_turns(pos, turns[lane + 32 * k]), &sr[k], &cr[k]);
  }
}

// The B fragments of the query columns for one stream, built by the warp from
// the raw query rows q[GS][D] (bf16, shared memory): column c = lane / 4 of
// the MMA is the head (c even) or the remainder (c odd) of query head c / 2
// (c < 2 GS), or zero; the angles each lane needs are shuffled in.  Lane (c, j =
// lane % 4) of k-step ks holds the elements d = 16 ks + {2j, 2j + 1, 2j + 8,
// 2j + 9} (bf16 cache: the MMA's own k order) or d = 16 ks + 4j + {0..3}
// (int8 cache: the k order of the K fragments the codes are unpacked into).
// Int8: the values are scaled by 2^kq so that the largest lies in
// [2^13, 2^14) (|q_rot| <= sqrt(2) max|q| bounds it: the rotation keeps each
// pair's norm); *inv_sq returns 2^-kq.
template <int D, int GS, bool INT8>
__device__ __forceinline__ void warp_query_fragments(const DecodeParams &p, const float (&cr)[D / 64],
                                                     const float (&sr)[D / 64],
                                                     const __nv_bfloat16 *qrows, int lane,
                                                     uint32_t (&qb)[D / 16][2], float &inv_sq) {
  constexpr int H = D / 2, KS = D / 16;
  constexpr int e2 = INT8 ? 2 : 8;  // offset of the fragment's second element pair
  const int col = lane >> 2;
  const bool used = col < 2 * GS;
  const bool is_lo = (col & 1) != 0;
  const int head = used ? col >> 1 : 0;
  const uint32_t *q32 = reinterpret_cast<const uint32_t *>(qrows + head * D);
  const int d0 = (INT8 ? 4 : 2) * (lane & 3);
  uint32_t w[KS / 2][4];  // raw pairs: (d, d+1), (d+e2, d+e2+1) and the same + H
#pragma unroll
  for (int kp = 0; kp < KS / 2; ++kp) {
    const int d = 16 * kp + d0;
    w[kp][0] = used ? q32[d / 2] : 0u;
    w[kp][1] = used ? q32[(d + e2) / 2] : 0u;
    w[kp][2] = used ? q32[(d + H) / 2] : 0u;
    w[kp][3] = used ? q32[(d + H + e2) / 2] : 0u;
  }
  float qs = p.qscale;
  inv_sq = 1.f;
  if constexpr (INT8) {
    uint32_t mx = 0;  // largest |q| as bf16 magnitude bits
#pragma unroll
    for (int kp = 0; kp < KS / 2; ++kp)
#pragma unroll
      for (int k = 0; k < 4; ++k) mx = max(mx, max(w[kp][k] & 0x7fffu, (w[kp][k] >> 16) & 0x7fffu));
    mx = __reduce_max_sync(0xffffffffu, mx);
    const float bound = __uint_as_float(mx << 16) * fabsf(p.qscale) * 1.4143f;
    const int eb = (int)((__float_as_uint(bound) >> 23) & 0xffu) - 127;
    const int kq = max(-100, min(100, 13 - eb));
    qs = p.qscale * pow2i(kq);
    inv_sq = pow2i(-kq);
  }
#pragma unroll
  for (int kp = 0; kp < KS / 2; ++kp) {
    // elements d + {0, 1, e2, e2 + 1} of the first half and the same + H of
    // the second half of each rotation pair; their angles live in register
    // (16 kp) / 32 of lanes (d + e) % 32
    const int d = 16 * kp + d0;
    const int reg = (16 * kp) / 32;
    const int e[4] = {0, 1, e2, e2 + 1};
    float c[4], s[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int src = (d + e[k]) & 31;
      c[k] = __shfl_sync(0xffffffffu, pick(cr, reg), src);
      s[k] = __shfl_sync(0xffffffffu, pick(sr, reg), src);
    }
    const float2 a0 = bf16x2_to_float2(w[kp][0]), a1 = bf16x2_to_float2(w[kp][1]);
    const float2 b0 = bf16x2_to_float2(w[kp][2]), b1 = bf16x2_to_float2(w[kp][3]);
    const float lo[4] = {a0.x, a0.y, a1.x, a1.y};
    const float hi[4] = {b0.x, b0.y, b1.x, b1.y};
    float vl[4], vh[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      vl[k] = (lo[k] * c[k] - hi[k] * s[k]) * qs;
      vh[k] = (hi[k] * c[k] + lo[k] * s[k]) * qs;
      const float tl = INT8 ? f16_round(vl[k]) : bf16_round(vl[k]);
      const float th = INT8 ? f16_round(vh[k]) : bf16_round(vh[k]);
      vl[k] = is_lo ? vl[k] - tl : tl;
      vh[k] = is_lo ? vh[k] - th : th;
    }
    if constexpr (INT8) {
      qb[kp][0] = pack_f16(vl[0], vl[1]);
      qb[kp][1] = pack_f16(vl[2], vl[3]);
      qb[kp + KS / 2][0] = pack_f16(vh[0], vh[1]);
      qb[kp + KS / 2][1] = pack_f16(vh[2], vh[3]);
    } else {
      qb[kp][0] = pack_bf16(vl[0], vl[1]);
      qb[kp][1] = pack_bf16(vl[2], vl[3]);
      qb[kp + KS / 2][0] = pack_bf16(vh[0], vh[1]);
      qb[kp + KS / 2][1] = pack_bf16(vh[2], vh[3]);
    }
  }
}

// Lines per CTA of an L2 prefetch spread over the grid: an fp32 estimate of
// lines / grid plus two.  A prefetch is only a hint (a line fetched twice
// costs little, one left out only waits later), and the CTAs placed last run
// this before their wait, on the step's critical path: no 64-bit division.
__device__ __forceinline__ size_t prefetch_share(size_t lines) {
  float rg;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(rg) : "f"((float)gridDim.x));
  return (size_t)((float)lines * rg) + 2;
}

// KV head of stream si of a sequence (n_sub query-head groups per KV head);
// most models have one group per KV head, which skips the division
__device__ __forceinline__ int sub_head(int si, int n_sub) { return n_sub == 1 ? si : si / n_sub; }

template <int D, int GS, bool INT8, bool LAYERED>
// at most 3 CTAs fit an SM's shared memory: let each thread have 1/384 of the
// register file
__global__ void __launch_bounds__(kDecodeThreads, 3)
    decode_mma_kernel(const __grid_constant__ DecodeParams p) {
  using C = MmaCfg<D, GS, INT8>;
  constexpr int W = C::W;
  const float kNegInf = -INFINITY;
  const float kFloor = -1e30f;  // initial reference maximum, below any score
  const float kLazy = 8.f;      // log2 headroom of the lazy softmax references
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint8_t *stages = smem;
  float *scales = reinterpret_cast<float *>(smem + C::kScaleOff);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kBarOff);
  float2 *turns = reinterpret_cast<float2 *>(smem + C::kFreqOff);
  double *inv_freq = reinterpret_cast<double *>(smem + C::kInvOff);
  int *misc = reinterpret_cast<int *>(smem + C::kMiscOff);
  float4 *angle_tab = reinterpret_cast<float4 *>(smem + C::kTabOff);
  int *pref = reinterpret_cast<int *>(smem + C::kPrefOff);
  int *lens = pref + p.n_seq + 1;
  int *poss = lens + p.n_seq;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  __nv_bfloat16 *qbuf = reinterpret_cast<__nv_bfloat16 *>(smem + C::kQOff) + warp * GS * D;
  // physical page of each stage's unit (-1: out of range, the unit is skipped)
  volatile int *spage = reinterpret_cast<int *>(smem + C::kValidOff) + warp * C::kSW;
  const int spu = p.n_kvh * p.n_sub;
  // set-up that reads nothing an earlier kernel writes (launched as a
  // programmatic dependent, the grid may start before that kernel ends):
  // the frequency tables go to shared memory (lanes index them by pair, and
  // divergent reads of kernel parameters serialise), and so does the sin/cos
  // step table; the stage barriers are initialised
  if (tid < D / 2) {
    turns[tid] = p.turns[tid];
    inv_freq[tid] = p.inv_freq[tid];
  }
  for (int i = tid; i < C::kTabBytes / 16; i += kDecodeThreads) angle_tab[i] = kSinCosStep[i];
  if (tid == 0) {
    for (int s = 0; s < W * C::kSW; ++s) mbar_init(&bars[s], 1);
    for (int w = 0; w < W; ++w) mbar_init(reinterpret_cast<uint64_t *>(smem + C::kMiscOff + 32) + w, 1);
#ifdef KVATTN_TEST_STALL
    mbar_init(reinterpret_cast<uint64_t *>(smem + C::kMiscOff + 16), 1);  // never arrived at
#endif
    fence_barrier_init();
    prefetch_tensormap(&p.tmap_k);
    prefetch_tensormap(&p.tmap_v);
  }
  {
    // L2 prefetches of the step's small inputs, issued before the wait on the
    // previous kernel so that their address translations and DRAM reads
    // overlap its end.  A prefetch consumes nothing: L2 is the GPU's point of
    // coherence, so a line the previous kernel writes afterwards is updated
    // there, and every read of these inputs comes after the wait.
    // The lengths and positions, which every CTA reads first:
    const int n_len_lines = (p.n_seq * 4 + 127) / 128;
    for (int l = tid; l < n_len_lines; l += kDecodeThreads) {
      asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char *>(p.seq_lens) + l * 128));
      asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char *>(p.positions) + l * 128));
    }
    // every CTA pulls its slice of the queries into L2, so that the warps'
    // query rows do not queue behind the flood of K/V requests
    const size_t q_lines = ((size_t)p.n_layers * p.n_seq * p.n_qh * D * 2 + 127) / 128;
    const size_t per = prefetch_share(q_lines);
    const char *qc = reinterpret_cast<const char *>(p.q);
#pragma unroll 1
    for (size_t l = blockIdx.x * per + tid; l < min(q_lines, (blockIdx.x + 1) * per); l += kDecodeThreads)
      asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(qc + l * 128));
    // and the new keys and values, which the warps appending them read
    const size_t kv_lines = ((size_t)p.n_layers * p.n_seq * p.n_kvh * D * 2 + 127) / 128;
    const size_t kper = prefetch_share(kv_lines);
    const char *kc = reinterpret_cast<const char *>(p.k_new);
    const char *vc = reinterpret_cast<const char *>(p.v_new);
#pragma unroll 1
    for (size_t l = blockIdx.x * kper + tid; l < min(kv_lines, (blockIdx.x + 1) * kper);
         l += kDecodeThreads) {
      asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(kc + l * 128));
      asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(vc + l * 128));
    }
    // and the block table when it is small, so that the page look-ups after
    // the planning below find it in L2 instead of waiting on DRAM again
    const size_t bt_lines = ((size_t)p.n_seq * p.max_pages * 4 + 127) / 128;
    if (bt_lines <= kTablePrefetchLines) {
      const size_t bper = prefetch_share(bt_lines);
      const char *bc = reinterpret_cast<const char *>(p.block_table);
#pragma unroll 1
      for (size_t l = blockIdx.x * bper + tid; l < min(bt_lines, (blockIdx.x + 1) * bper); l += kDecodeThreads)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(bc + l * 128));
    }
  }
  pdl_wait_primary();       // every earlier kernel of the stream is complete and visible
  pdl_launch_dependents();  // the combine grid may start planning at once
  // prefix sums of units per sequence, lengths and positions (its barriers
  // also publish the set-up above); shares are per warp here
  int TL = 0;  // units of one layer
  if (!plan_units<kDecodeThreads>(p, pref, misc, TL, lens, poss, blockIdx.x == 0)) return;
  const int n_warps = min((int)gridDim.x * W, p.n_shares);
  // (LAYERED: the call decodes several layer caches, else one)
  const int n_layers = LAYERED ? p.n_layers : 1;
  const int nwa = warp_shares(n_layers * (4 * TL + p.stream_cost * p.n_seq * spu), n_warps);
  const WeightedSplit split(pref, p.n_seq, spu, p.stream_cost, TL, n_layers, nwa);
  const auto rope_of = [&](int l) { return LAYERED ? layer_rope(p, l) : p.use_rope != 0; };
  // A small batch leaves at least half of the warps idle: then the shares
  // are spread over the CTAs (warp slots 0..A-1 of every CTA; A <= W/2) and
  // idle warp A + a of a CTA forms the new token's stored row of active warp
  // a's first stream, if a appends it, while a streams its units (a warp
  // alone takes microseconds for the correctly rounded cos/sin).  Otherwise
  // warp g of the grid takes share g.
  const bool spread = 2 * nwa <= n_warps;
  // (spread: nwa <= grid W / 2, so A = ceil(nwa / grid) is 1 or 2)
  static_assert(W == 4, "two spread shares per CTA at most");
  const int A = spread ? (nwa > (int)gridDim.x ? 2 : 1) : W;
  const int g = spread ? warp * (int)gridDim.x + (int)blockIdx.x : (int)blockIdx.x * W + warp;
  uint64_t *row_ready = reinterpret_cast<uint64_t *>(smem + C::kMiscOff + 32);  // [W]
  if (g >= nwa) {
    const int a = warp - A;
    const int ga = a * (int)gridDim.x + (int)blockIdx.x;
    if (spread && a >= 0 && a < A && ga < nwa) {
      int b = 0, b1 = 0, wa0 = 0, wa1 = 0;
      split.share_bounds<LAYERED>(ga, lane, &wa0, &b, &wa1, &b1);
      if (wa0 >= wa1) b = 0;
      const UnitPos up = locate_unit<LAYERED>(wa0 < wa1 ? wa0 : 0, b, pref, spu, p.n_seq, TL);
      if (wa0 < wa1 && up.first + up.units <= wa1) {  // warp a appends its first stream's new token
        uint8_t *arow = smem + C::kNewOff + a * C::kNewBytes;
        const size_t kv = ((size_t)up.v * p.n_kvh + sub_head(up.si, p.n_sub)) * D;
        const char *ks = reinterpret_cast<const char *>(p.k_new + kv);
        const char *vs = reinterpret_cast<const char *>(p.v_new + kv);
        for (int c = lane; c < 4 * D / 16; c += 32)
          cp_async_16(arow + c * 16, (c < 2 * D / 16 ? ks + c * 16 : vs + (c - 2 * D / 16) * 16));
        cp_async_wait_all();
        __syncwarp();
        stage_new_row<D, INT8>(poss[up.b], inv_freq, angle_tab, rope_of(up.l), lane, arow);
        if (lane == 0) mbar_arrive(&row_ready[a]);  // (release: the row is visible)
      }
    }
    return;
  }
  int start_v = 0, end_v = 0, wt0 = 0, wt1 = 0;
  split.share_bounds<LAYERED>(g, lane, &wt0, &start_v, &wt1, &end_v);
  const int count = wt1 - wt0;
  if (count == 0) return;  // a share of stream costs only
  const uint64_t pol = l2_evict_first_policy();

  // raw query rows of a stream -> this warp's buffer by 16-byte cp.async (an
  // LSU copy from L2, where the prologue put the queries: a bulk copy would
  // queue behind the SM's flood of tile copies).  With the int8 cache, lanes
  // 0-7 issue the scale copies that the stage barriers track, so only lanes
  // kQLane0.. copy (and wait for) query rows.
  constexpr int kQLane0 = INT8 ? 8 : 0;
  auto prefetch_queries = [&](int v, int h0) {  // (virtual sequence v)
    __syncwarp();
    const char *src = reinterpret_cast<const char *>(p.q + ((size_t)v * p.n_qh + h0) * D);
    if (lane >= kQLane0)
      for (int c = lane - kQLane0; c < C::kQBytes / 16; c += 32 - kQLane0)
        cp_async_16(reinterpret_cast<char *>(qbuf) + c * 16, src + c * 16);
    cp_async_commit();
  };
  // raw new key and value rows of (sequence b, KV head j) -> the warp's
  // new-row buffer, the same way (any plain load issued once the SM's inbound
  // queue is full of tiles waits microseconds behind them)
  uint8_t *nrow = smem + C::kNewOff + warp * C::kNewBytes;
  auto prefetch_new_raw = [&](int v, int j) {
    const size_t kv = ((size_t)v * p.n_kvh + j) * D;
    const char *ks = reinterpret_cast<const char *>(p.k_new + kv);
    const char *vs = reinterpret_cast<const char *>(p.v_new + kv);
    if (lane >= kQLane0)
      for (int c = lane - kQLane0; c < 4 * D / 16; c += 32 - kQLane0)
        cp_async_16(nrow + c * 16, (c < 2 * D / 16 ? ks + c * 16 : vs + (c - 2 * D / 16) * 16));
    cp_async_commit();
  };
  // position of the next unit to request: layer, sequence, KV head,
  // query-head group and unit of the stream, advanced one unit at a time by
  // every lane alike
  int cb_l, cb_b, cb_j, cb_sub, cb_u, cb_units;
  {
    int v = start_v;
    const UnitPos up = locate_unit<LAYERED>(wt0, v, pref, spu, p.n_seq, TL);
    cb_l = up.l;
    cb_b = up.b;
    cb_j = sub_head(up.si, p.n_sub);
    cb_sub = up.si - cb_j * p.n_sub;
    cb_u = up.u;
    cb_units = up.units;
    prefetch_queries(up.v, cb_j * GS * p.n_sub + cb_sub * GS);
    // the first stream's raw new rows, if this warp appends it and no idle
    // warp does the work
    if (up.first + up.units <= wt1 && !(spread && warp + A < W)) prefetch_new_raw(up.v, cb_j);
  }
  auto advance = [&]() {  // only while units remain in the share
    if (++cb_u < cb_units) return;
    cb_u = 0;
    if (++cb_sub < p.n_sub) return;
    cb_sub = 0;
    if (++cb_j < p.n_kvh) return;
    cb_j = 0;
    do {
      ++cb_b;
      if (LAYERED && cb_b == p.n_seq) {
        cb_b = 0;
        ++cb_l;
      }
    } while (pref[cb_b + 1] == pref[cb_b]);
    cb_units = pref[cb_b + 1] - pref[cb_b];
  };

  // ---- producer ---------------------------------------------------------------
  // Physical pages are fetched 32 units ahead, one per lane, so the issuing
  // lane never waits on the block table.  The last unit of a stream holds the
  // slot of the new token, which the warp consuming that unit fills in shared
  // memory itself (below): nothing waits for the pool write.
  // (raw block-table entries: the range check waits until a page is used, so
  // that the second window's load does not stall the first requests)
  int pcur = start_v;  // per-lane cursor of the page windows
  int win_base = 0;
  int win_page = lane < count ? page_raw_of_unit<LAYERED>(p, pref, spu, TL, wt0 + lane, pcur) : -1;
  int nxt_page = 32 + lane < count ? page_raw_of_unit<LAYERED>(p, pref, spu, TL, wt0 + 32 + lane, pcur) : -1;
  auto issue = [&](int i) {  // called by the whole warp, in unit order
    if (i > 0) advance();
    if (i - win_base >= 32) {
      win_base += 32;
      win_page = nxt_page;
      const int tn = win_base + 32 + lane;
      nxt_page = tn < count ? page_raw_of_unit<LAYERED>(p, pref, spu, TL, wt0 + tn, pcur) : -1;
    }
    int page = __shfl_sync(0xffffffffu, win_page, i - win_base);
    // range-checked in its layer's pool, then a page of the all-layer view
    page = (page >= 0 && page < p.num_pages) ? page + (LAYERED ? cb_l * p.num_pages : 0) : -1;
    const int st = warp * C::kSW + i % C::kSW;
    const int row = (page * p.n_kvh + cb_j) * p.page_size + ((cb_u * kUnitRows) & (p.page_size - 1));
    if constexpr (INT8) {
      // the unit's 2 x 64 bytes of row scales: one 16-byte cp.async per lane
      // 0-7, which the stage's barrier tracks (each raises the barrier's
      // pending count until its copy lands, before lane 0 arrives below)
      if (page >= 0 && lane < 8) {
        cp_async_16(scales + st * (2 * kUnitRows) + 4 * lane,
                    (lane < 4 ? p.k_scales : p.v_scales) + row + 4 * (lane & 3));
        cp_async_mbar_arrive(&bars[st]);
      }
      __syncwarp();
    }
    if (lane == 0) {
      spage[i % C::kSW] = page;
      if (page >= 0) {
        uint8_t *dst = stages + (size_t)st * C::kStage;
        mbar_arrive_expect_tx(&bars[st], C::kStage);
#pragma unroll
        for (int r = 0; r < C::kRegions; ++r) {
          const int x = r * C::kBoxW / (INT8 ? 1 : 2);  // element column of box r
          tma_load_2d(dst + r * C::kBox, &p.tmap_k, x, row, &bars[st], pol);
          tma_load_2d(dst + C::kTile + r * C::kBox, &p.tmap_v, x, row, &bars[st], pol);
        }
      } else {
        atomicOr(p.status, KVATTN_DEV_BAD_PAGE);
        mbar_arrive(&bars[st]);
      }
    }
  };
  int issued = 0;
  for (; issued < min(C::kSW, count); ++issued) issue(issued);

  // ---- consumer ---------------------------------------------------------------
  // this lane's score and output columns are 2 hl (head) and 2 hl + 1
  // (remainder) of query head hl; lanes with hl >= GS hold padding columns
  const int hl = lane & 3;
  const int tokr = lane >> 2;                     // this lane's score rows: tokr, tokr + 8
  // ldmatrix row addresses: K (and int8 V) read matrices (rows 0-7, chunk c),
  // (rows 8-15, c), (rows 0-7, c + 1), (rows 8-15, c + 1); bf16 V, transposed,
  // reads (rows 0-7, c), (rows 0-7, c + 1), (rows 8-15, c), (rows 8-15, c + 1)
  const int krow = (lane & 7) + ((lane >> 3) & 1) * 8, kcsel = lane >> 4;
  const int vrow = INT8 ? krow : (lane & 7) + (lane >> 4) * 8;
  const int vcsel = INT8 ? kcsel : (lane >> 3) & 1;
  bool aborted = false;
#ifdef KVATTN_TEST_STALL
  if ((__ldcg(p.status) & kTestStallRequest) != 0 &&
      !__all_sync(0xffffffffu, mbar_wait_bounded(reinterpret_cast<uint64_t *>(smem + C::kMiscOff + 16),
                                                  0, kTestStallCycles))) {
    aborted = true;
    if (lane == 0) atomicOr(p.status, KVATTN_DEV_TIMEOUT);
  }
#endif
  int consumed = 0;
  int cb = start_v;
  int t = wt0;
  while (t < wt1) {
    const UnitPos sp = locate_unit<LAYERED>(t, cb, pref, spu, p.n_seq, TL);
    const int F = sp.first, E = F + sp.units;
    const int e = min(wt1, E);
    const int L = lens[sp.b];
    const int j = sub_head(sp.si, p.n_sub), sub = sp.si - j * p.n_sub;
    const int h0 = j * GS * p.n_sub + sub * GS;
    const int sid = sp.v * spu + sp.si;  // (all layers' streams)

    // The warp that consumes the stream's last unit forms the stored key and
    // value of the new token (the storage recipe, storage.cuh) once that
    // unit's copy is in flight (kSW units ahead), while it waits for data
    // anyway; when the tile has landed it puts them into the tile in place of
    // whatever the pool held in the slot, and writes them to slot L of the
    // pool (for the KV head's first query-head group only: one writer per
    // slot).  So the step's attention never waits for its own append.
    const bool own_last = E <= wt1;
    const bool helped = own_last && t == wt0 && spread && warp + A < W;  // row formed by a helper
    const int tab_at = max(t, E - C::kSW);

    uint32_t qb[C::kKSteps][2];
    float inv_sq;
    float cr[D / 64], sr[D / 64];
    warp_query_angles<D>(turns, poss[sp.b], rope_of(sp.l), lane, cr, sr);  // while the rows land
    if (lane >= kQLane0) cp_async_wait_all();
    __syncwarp();
    warp_query_fragments<D, GS, INT8>(p, cr, sr, qbuf, lane, qb, inv_sq);
    __syncwarp();
    // int8: the key codes enter the MMA as 1152 + x; -1152 * (column sum of
    // Qc), formed by the same MMA with a constant A of -1152, is where every
    // unit's dot products start (this lane's columns 2 (lane % 4) + {0, 1})
    float kbias[2] = {0.f, 0.f};
    if constexpr (INT8) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      const uint32_t m1152[4] = {0xe480e480u, 0xe480e480u, 0xe480e480u, 0xe480e480u};
#pragma unroll
      for (int ks = 0; ks < C::kKSteps; ++ks) mma_f16_16816(acc, m1152, qb[ks][0], qb[ks][1]);
      kbias[0] = acc[0];
      kbias[1] = acc[1];
    }
    if (E < wt1) {  // the share continues: fetch the next stream's query rows
      int v = sp.v;
      const UnitPos nx = locate_unit<LAYERED>(E, v, pref, spu, p.n_seq, TL);
      const int nj = sub_head(nx.si, p.n_sub);
      prefetch_queries(nx.v, nj * GS * p.n_sub + (nx.si - nj * p.n_sub) * GS);
    }
    // this stream's raw new rows (the first stream's came in the prologue),
    // after the query wait above so that it does not wait for them
    if (own_last && t > wt0) prefetch_new_raw(sp.v, j);
    float o[C::kKSteps][4];
#pragma unroll
    for (int dt = 0; dt < C::kKSteps; ++dt)
#pragma unroll
      for (int k = 0; k < 4; ++k) o[dt][k] = 0.f;
    // m, l: reference maximum and normaliser of the softmax of head hl; dmo:
    // reference maximum of its value weights, less m (int8; the bf16 cache
    // weighs the values by the softmax weights themselves).  The references
    // start at a finite floor below every score, so no step needs a guard for
    // an empty state.
    float m = kFloor, l = 0.f, dmo = kFloor;

    for (int tt = t; tt < e; ++tt) {
      if (own_last && tt == tab_at && !helped) {
        if (lane >= kQLane0) cp_async_wait_all();  // the raw rows
        __syncwarp();
        stage_new_row<D, INT8>(poss[sp.b], inv_freq, angle_tab, rope_of(sp.l), lane, nrow);
      }
      const int i = (int)(tt - wt0);
      const int st = warp * C::kSW + i % C::kSW;
      bool ok = false;
      if (!aborted) {
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars[st], (uint32_t)((i / C::kSW) & 1)));
        if (!ok) {
          aborted = true;
          if (lane == 0) atomicOr(p.status, KVATTN_DEV_TIMEOUT);
        }
        consumed = i + 1;  // stages waited for (or given up on) so far
      }
      const int tok0 = (int)(tt - F) * kUnitRows;
      const int upage = spage[i % C::kSW];
      if (ok && upage >= 0) {
        const int nrows = min(kUnitRows, L + 1 - tok0);
        uint8_t *Ks = stages + (size_t)st * C::kStage;
        uint8_t *Vs = Ks + C::kTile;
        const uint32_t kb = smem_addr(Ks), vb = smem_addr(Vs);
        if (own_last && tt == E - 1) {  // slot L is row L - tok0 of the last unit
          if (helped && !__all_sync(0xffffffffu, mbar_wait_bounded(&row_ready[warp], 0))) {
            aborted = true;
            if (lane == 0) atomicOr(p.status, KVATTN_DEV_TIMEOUT);
          }
          const long long slot =
              sub == 0 ? ((long long)upage * p.n_kvh + j) * p.page_size + (L & (p.page_size - 1)) : -1;
          put_new_row<D, INT8>(nrow, Ks, Vs, scales + st * (2 * kUnitRows), L - tok0, slot,
                               p.k_pages, p.v_pages, p.k_scales, p.v_scales, lane,
                               [](int r, int ch) { return tile_off<C>(r, ch); });
          __syncwarp();
        }
        if (!INT8 && nrows < kUnitRows) {
          // bf16 rows past the sequence end hold stale data: zero them in V
          // so that their zero weights cannot meet a NaN (int8 codes are
          // always finite)
          const int n16 = (kUnitRows - nrows) * C::kRegions * 8;
          for (int idx = lane; idx < n16; idx += 32) {
            const int row = nrows + idx / (C::kRegions * 8);
            const int c = idx % (C::kRegions * 8);
            *reinterpret_cast<uint4 *>(Vs + (c >> 3) * C::kBox + row * 128 + (c & 7) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          __syncwarp();
        }
        // int8: scale of this lane's score rows (with the query's 2^-kq) and
        // log2 of the value scales
        float ksr[2] = {1.f, 1.f}, lv[2] = {0.f, 0.f};
        if constexpr (INT8) {
          const float *sc = scales + st * (2 * kUnitRows);
#pragma unroll
          for (int t2 = 0; t2 < 2; ++t2) {
            ksr[t2] = sc[tokr + 8 * t2] * inv_sq;
            lv[t2] = lg2_approx(sc[kUnitRows + tokr + 8 * t2]);
          }
        }

        // S^T = K Qc^T (int8: from -1152 * column sums of Qc, see kbias)
        float s[4] = {kbias[0], kbias[1], kbias[0], kbias[1]};
#pragma unroll
        for (int it = 0; it < C::kLdm; ++it) {
          uint32_t a[4];
          ldmatrix_x4(a, kb + tile_off<C>(krow, 2 * it + kcsel));
          if constexpr (INT8) {
            // codes of rows g, g + 8 at d = 4j..4j+3 of chunks 2 it, 2 it + 1:
            // k-step 2 it + c takes (d 4j, 4j+1) as its columns 2j, 2j+1 and
            // (4j+2, 4j+3) as 2j+8, 2j+9, matching the query fragments
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              const uint32_t r0 = a[2 * c] ^ 0x80808080u, r1 = a[2 * c + 1] ^ 0x80808080u;
              const uint32_t f[4] = {codes_biased_f16x2(r0, 0x5140u),
                                     codes_biased_f16x2(r1, 0x5140u),
                                     codes_biased_f16x2(r0, 0x5342u),
                                     codes_biased_f16x2(r1, 0x5342u)};
              mma_f16_16816(s, f, qb[2 * it + c][0], qb[2 * it + c][1]);
            }
          } else {
            mma_bf16_16816(s, a, qb[it][0], qb[it][1]);
          }
        }
        // full scores of head hl at tokens tokr, tokr + 8: head column plus
        // remainder column
        float sc[2] = {s[0] + s[1], s[2] + s[3]};
        if constexpr (INT8) {
          sc[0] *= ksr[0];
          sc[1] *= ksr[1];
        }
        if (nrows < kUnitRows) {  // a sequence's last unit: drop the rows past its end
#pragma unroll
          for (int t2 = 0; t2 < 2; ++t2)
            if (tokr + 8 * t2 >= nrows) sc[t2] = lv[t2] = kNegInf;  // (stale scales too)
        }

        // online softmax (log2 units) with lazy references: a reference moves
        // only when a score passes it by more than kLazy, so every weight stays
        // below 2^kLazy and most units leave the accumulators as they are
        float pv[2];
        float alpha = 1.f;
        {
          float mx = fmaxf(sc[0], sc[1]);
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          float a = 1.f;
          if (mx > m + kLazy) {
            a = ex2_approx(m - mx);
            if constexpr (INT8) dmo -= mx - m;  // the same absolute reference
            m = mx;
          }
          const float pw0 = ex2_approx(sc[0] - m), pw1 = ex2_approx(sc[1] - m);
          l = l * a + pw0 + pw1;
          if constexpr (INT8) {
            // value-weight exponents S - m + log2 vs: log2 vs is added to a
            // number near zero, so fp32 keeps it whatever the scores' size
            const float xv0 = (sc[0] - m) + lv[0], xv1 = (sc[1] - m) + lv[1];
            float xo = fmaxf(xv0, xv1);
            xo = fmaxf(xo, __shfl_xor_sync(0xffffffffu, xo, 4));
            xo = fmaxf(xo, __shfl_xor_sync(0xffffffffu, xo, 8));
            xo = fmaxf(xo, __shfl_xor_sync(0xffffffffu, xo, 16));
            a = 1.f;
            if (xo > dmo + kLazy) {
              a = ex2_approx(dmo - xo);
              dmo = xo;
            }
            pv[0] = ex2_approx(xv0 - dmo);
            pv[1] = ex2_approx(xv1 - dmo);
          } else {
            pv[0] = pw0;
            pv[1] = pw1;
          }
          alpha = a;
        }
        // P^T fragments: this lane's two columns at tokens tokr and tokr + 8:
        // the value weight rounded to the MMA's type and what that rounding
        // left out
        uint32_t pr[2];
#pragma unroll
        for (int t2 = 0; t2 < 2; ++t2) {
          const float hi = INT8 ? f16_round(pv[t2]) : bf16_round(pv[t2]);
          pr[t2] = INT8 ? pack_f16(hi, pv[t2] - hi) : pack_bf16(hi, pv[t2] - hi);
        }
        const uint32_t b0 = movmatrix_trans(pr[0]);
        const uint32_t b1 = movmatrix_trans(pr[1]);
        // rescale the accumulators of this lane's columns when a reference moved
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int dt = 0; dt < C::kKSteps; ++dt)
#pragma unroll
            for (int k = 0; k < 4; ++k) o[dt][k] *= alpha;
        }
        // O^T += V^T P^T
#pragma unroll
        for (int it = 0; it < C::kLdm; ++it) {
          uint32_t a[4];
          ldmatrix_x4_trans(a, vb + tile_off<C>(vrow, 2 * it + vcsel));
          if constexpr (INT8) {
            // lane (g, j) holds codes of tokens 2j, 2j+1 (rows 0-7: a[2c],
            // rows 8-15: a[2c+1]) at d = 2g, 2g+1 of chunk 2 it + c: m-tile
            // row g takes d = 2g, row g + 8 takes d = 2g + 1
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              const uint32_t r0 = a[2 * c] ^ 0x80808080u, r1 = a[2 * c + 1] ^ 0x80808080u;
              const uint32_t f[4] = {codes_to_f16x2(r0, 0x5240u), codes_to_f16x2(r0, 0x5341u),
                                     codes_to_f16x2(r1, 0x5240u), codes_to_f16x2(r1, 0x5341u)};
              mma_f16_16816(o[2 * it + c], f, b0, b1);
            }
          } else {
            mma_bf16_16816(o[it], a, b0, b1);
          }
        }
      }
      __syncwarp();
      if (!aborted && issued < count) {
        if (lane == 0) fence_proxy_async_smem();
        issue(issued);
        ++issued;
      }
    }

    // ---- end of this warp's part of the stream ----------------------------------
    // head column plus remainder column; l summed over the tokens
    float of[C::kKSteps][2];
#pragma unroll
    for (int dt = 0; dt < C::kKSteps; ++dt) {
      of[dt][0] = o[dt][0] + o[dt][1];
      of[dt][1] = o[dt][2] + o[dt][3];
    }
    l += __shfl_xor_sync(0xffffffffu, l, 4);
    l += __shfl_xor_sync(0xffffffffu, l, 8);
    l += __shfl_xor_sync(0xffffffffu, l, 16);
    // accumulator scale to 2^m (int8: from 2^(m + dmo))
    const float to_m = INT8 ? ex2_approx(dmo) : 1.f;
    // lanes with hl < GS hold head hl's output rows d = dA(dt) (of[dt][0])
    // and d = dB(dt) (of[dt][1])
    const bool writer = hl < GS;
    const int dr = lane >> 2;
    const auto dA = [&](int dt) { return INT8 ? dt * 16 + 2 * dr : dt * 16 + dr; };
    const auto dB = [&](int dt) { return INT8 ? dt * 16 + 2 * dr + 1 : dt * 16 + dr + 8; };
    __nv_bfloat16 *outp = p.out + ((size_t)sp.v * p.n_qh + h0 + hl) * D;
    if (F >= wt0 && E <= wt1) {
      if (writer) {
        const float f = l > 0.f ? to_m / l : 0.f;
#pragma unroll
        for (int dt = 0; dt < C::kKSteps; ++dt) {
          outp[dA(dt)] = __float2bfloat16_rn(of[dt][0] * f);
          outp[dB(dt)] = __float2bfloat16_rn(of[dt][1] * f);
        }
      }
    } else {
      // partial record of this warp's part: acc[GS][D] relative to 2^m, m, l
      // (the records of a stream's parts are consecutive: one slot per share)
      float *rec = p.records + (size_t)(sid + g) * C::RS;
      if (writer) {
#pragma unroll
        for (int dt = 0; dt < C::kKSteps; ++dt) {
          rec[hl * D + dA(dt)] = of[dt][0] * to_m;
          rec[hl * D + dB(dt)] = of[dt][1] * to_m;
        }
        if (dr == 0) {
          rec[GS * D + hl] = m;
          rec[GS * D + GS + hl] = l;
        }
      }
    }
    t = e;
  }

  cp_async_wait_all();  // no copy may land after the warp has left
  if (aborted && lane == 0) {
    // copies issued to stages no wait has looked at since are still in
    // flight: let them land before the warp leaves
    for (int i = consumed; i < issued; ++i)
      (void)mbar_wait_bounded(&bars[warp * C::kSW + i % C::kSW], (uint32_t)((i / C::kSW) & 1));
  }
}

template <int D, int GS, bool INT8, bool LAYERED>
cudaError_t launch_decode_mma_t(const DecodeParams &p, int grid, cudaStream_t stream,
                                int *ctas_per_sm, bool launch) {
  using C = MmaCfg<D, GS, INT8>;
  auto kern = decode_mma_kernel<D, GS, INT8, LAYERED>;
  const int smem = C::kFixedSmem + (int)align_up((size_t)(3 * p.n_seq + 1) * 4, 16);
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
                                 C::kFixedSmem + (3 * KVATTN_MAX_SEQS + 1) * 4 + 16);
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
  // a programmatic dependent of the stream's previous kernel: the grid may be
  // placed while that kernel finishes, and waits for it (griddepcontrol.wait)
  // before it reads or writes anything in global memory
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace kvattn
