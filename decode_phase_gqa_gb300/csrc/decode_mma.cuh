// Split-KV flash-decoding kernel for the bf16 KV cache, tensor-core inner loop.
//
// Work split.  Every (sequence, KV head, query-head group) is a stream of
// 16-token units; the streams are laid end to end and the flattened unit list
// is cut into equal contiguous shares, one per WARP of the grid.  Warps are
// independent after the CTA's prologue (the per-sequence prefix sums): each
// streams its share through its own ring of shared-memory stages filled by TMA
// tensor copies (cp.async.bulk.tensor.2d, [16 rows][64 columns] boxes, 128-byte
// swizzle so the ldmatrix reads below hit all 32 banks), keeps its softmax
// state in registers, and at each stream boundary either writes the output (a
// stream inside its share) or a partial record that the combine kernel
// (combine.cu, launched as this grid's programmatic dependent) merges.
//
// Per unit the warp computes, with m16n8k16 bf16 MMAs (fp32 accumulate):
//   S^T[16 tokens][8] = K[16][d] * Qc^T[d][8]
//   O^T[d][8]        += V^T[d][16] * P^T[16][8]
// The 8 MMA columns carry, for the GS query heads of the group, the bf16 head
// of each value and its bf16 remainder (x = hi + lo), so neither the query nor
// the softmax weights lose precision to bf16 rounding: columns h and GS + h
// are added back together.  K and V themselves are bf16 in the cache, exact.
// Tokens are the MMA rows, so one K/V block serves every head of the group
// ("Qwen3-8B inference engine from scratch in C++/CUDA", section 4.4.2:
// read the group's KV once for all its query heads), and the online softmax
// ("LLM inference from smollm3.go", section "Self-attention") runs on the
// accumulator fragments in fp32, in log2 units.
#pragma once

#include <map>
#include <mutex>
#include <set>
#include <utility>

#include "decode_common.cuh"

namespace kvattn {

template <int D, int GS>
struct MmaCfg {
  static constexpr int W = kDecodeWarps;
  static constexpr int kRegions = D / 64;   // 64-column swizzled boxes per 16-row tile
  static constexpr int kBox = 16 * 64 * 2;  // bytes of one box (2 KB)
  static constexpr int kTile = kRegions * kBox;
  static constexpr int kStage = 2 * kTile;  // K then V
  static constexpr int kQBytes = GS * D * 2;  // one stream's raw query rows (bf16)
  // stages per warp: as many as fit a 75 KB CTA (3 CTAs per SM) next to the
  // barriers, frequency table, per-warp query buffers and stage flags, the
  // 1 KB alignment slack and a 2 KB allowance for the per-sequence arrays
  static constexpr int kOther = W * 8 * 8 + 512 + 64 + W * kQBytes + W * 8 * 4 + 1024;
  static constexpr int kSWFit = (kCtaSmemBudget - kOther - 2048) / (W * kStage);
  static constexpr int kSW = kSWFit > 8 ? 8 : kSWFit;
  static constexpr int kKSteps = D / 16;
  static constexpr int kHL = GS == 1 ? 1 : 2;  // query heads per lane
  static constexpr int kStagesBytes = W * kSW * kStage;
  static constexpr int kBarOff = kStagesBytes;
  static constexpr int kFreqOff = kBarOff + W * kSW * 8;  // rope turns per position, float2[D/2]
  static constexpr int kMiscOff = kFreqOff + 512;
  static constexpr int kQOff = kMiscOff + 64;             // [W][GS][D] bf16
  static constexpr int kValidOff = kQOff + W * kQBytes;   // [W][kSW] int
  static constexpr int kPrefOff = kValidOff + W * kSW * 4;
  // fixed part + alignment slack; the per-sequence arrays (prefix sums,
  // lengths, positions: 3 n_seq + 1 ints) follow
  static constexpr int kFixedSmem = kPrefOff + 1024;
  static constexpr int RS = record_floats(GS, D);
  static_assert(kStage % 1024 == 0, "swizzled boxes need 1024-byte alignment");
  static_assert(kSW >= 2, "need at least double buffering");
  static_assert(kQBytes % 16 == 0, "query rows are copied in 16-byte chunks");
};

// swizzled byte offset of 16-byte chunk `chunk` of tile row `row` (rows of
// 128 bytes; chunk index XOR row mod 8, the TMA 128-byte swizzle)
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t u) {
  return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}

// RoPE of the query, fp32 only (the query needs fp32 accuracy): lane l holds
// cos/sin of angles l + 32k of position `pos`, from frac_turns and sincospif.
// Then the B fragments of the query columns for one stream, built by the warp
// from the raw query rows q[GS][D] (bf16, shared memory): column c = lane / 4
// of the MMA is the bf16 head of query head c (c < GS), its bf16 remainder
// (GS <= c < 2 GS), or zero; the angles each lane needs are shuffled in.
template <int D>
__device__ __forceinline__ void warp_query_angles(const DecodeParams &p, const float2 *turns,
                                                  int pos, int lane, float (&cr)[D / 64],
                                                  float (&sr)[D / 64]) {
#pragma unroll
  for (int k = 0; k < D / 64; ++k) {
    cr[k] = 1.f;
    sr[k] = 0.f;
    if (p.use_rope) sincospif(2.f * frac_turns(pos, turns[lane + 32 * k]), &sr[k], &cr[k]);
  }
}

template <int D, int GS>
__device__ __forceinline__ void warp_query_fragments(const DecodeParams &p, const float (&cr)[D / 64],
                                                     const float (&sr)[D / 64],
                                                     const __nv_bfloat16 *qrows, int lane,
                                                     uint32_t (&qb)[D / 16][2]) {
  constexpr int H = D / 2, KS = D / 16;
  const int col = lane >> 2;
  const bool used = col < 2 * GS;
  const bool is_lo = col >= GS;
  const int head = used ? (is_lo ? col - GS : col) : 0;
  const uint32_t *q32 = reinterpret_cast<const uint32_t *>(qrows + head * D);
  const int d0 = 2 * (lane & 3);
#pragma unroll
  for (int kp = 0; kp < KS / 2; ++kp) {
    // elements 16 kp + d0 + {0, 1, 8, 9} (first half) and the same + H
    // (second half) of each rotation pair; their angles live in register
    // (16 kp) / 32 of lanes (16 kp + d0 + e) % 32
    const int d = 16 * kp + d0;
    const uint32_t l0 = used ? q32[d / 2] : 0u, l1 = used ? q32[(d + 8) / 2] : 0u;
    const uint32_t h0 = used ? q32[(d + H) / 2] : 0u, h1 = used ? q32[(d + H + 8) / 2] : 0u;
    const int reg = (16 * kp) / 32;
    const int e[4] = {0, 1, 8, 9};
    float c[4], s[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int src = (d + e[k]) & 31;
      c[k] = __shfl_sync(0xffffffffu, pick(cr, reg), src);
      s[k] = __shfl_sync(0xffffffffu, pick(sr, reg), src);
    }
    const float2 a0 = bf16x2_to_float2(l0), a1 = bf16x2_to_float2(l1);
    const float2 b0 = bf16x2_to_float2(h0), b1 = bf16x2_to_float2(h1);
    const float lo[4] = {a0.x, a0.y, a1.x, a1.y};
    const float hi[4] = {b0.x, b0.y, b1.x, b1.y};
    float vl[4], vh[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      vl[k] = (lo[k] * c[k] - hi[k] * s[k]) * p.qscale;
      vh[k] = (hi[k] * c[k] + lo[k] * s[k]) * p.qscale;
      const float tl = __bfloat162float(__float2bfloat16_rn(vl[k]));
      const float th = __bfloat162float(__float2bfloat16_rn(vh[k]));
      vl[k] = is_lo ? vl[k] - tl : tl;
      vh[k] = is_lo ? vh[k] - th : th;
    }
    qb[kp][0] = pack_bf16(vl[0], vl[1]);
    qb[kp][1] = pack_bf16(vl[2], vl[3]);
    qb[kp + KS / 2][0] = pack_bf16(vh[0], vh[1]);
    qb[kp + KS / 2][1] = pack_bf16(vh[2], vh[3]);
  }
}

template <int D, int GS>
__global__ void __launch_bounds__(kDecodeThreads)
    decode_mma_kernel(const __grid_constant__ DecodeParams p) {
  using C = MmaCfg<D, GS>;
  constexpr int W = C::W;
  const float kNegInf = -INFINITY;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint8_t *stages = smem;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kBarOff);
  float2 *turns = reinterpret_cast<float2 *>(smem + C::kFreqOff);
  int *misc = reinterpret_cast<int *>(smem + C::kMiscOff);
  int *pref = reinterpret_cast<int *>(smem + C::kPrefOff);
  int *lens = pref + p.n_seq + 1;
  int *poss = lens + p.n_seq;

  pdl_launch_dependents();  // the combine grid may start planning at once
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  {
    // every CTA pulls its slice of the queries into L2 at once, so that the
    // warps' query rows do not queue behind the flood of K/V requests
    const size_t q_lines = ((size_t)p.n_seq * p.n_qh * D * 2 + 127) / 128;
    const size_t per = (q_lines + gridDim.x - 1) / gridDim.x;
    const char *qc = reinterpret_cast<const char *>(p.q);
    for (size_t l = blockIdx.x * per + tid; l < min(q_lines, (blockIdx.x + 1) * per); l += kDecodeThreads)
      asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(qc + l * 128));
  }
  __nv_bfloat16 *qbuf = reinterpret_cast<__nv_bfloat16 *>(smem + C::kQOff) + warp * GS * D;
  volatile int *svalid = reinterpret_cast<int *>(smem + C::kValidOff) + warp * C::kSW;
  const int spu = p.n_kvh * p.n_sub;
  if (tid < D / 2) turns[tid] = p.turns[tid];
  if (tid == 0) {
    for (int s = 0; s < W * C::kSW; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
    prefetch_tensormap(&p.tmap_k);
    prefetch_tensormap(&p.tmap_v);
  }
  // prefix sums of units per sequence, lengths and positions (its barriers
  // also publish the above); shares are per warp here
  long long T = 0;
  if (!plan_units<kDecodeThreads>(p, pref, misc, T, lens, poss)) return;
  const long long n_warps = min((long long)gridDim.x * W, (long long)p.n_shares);
  const long long nwa = min(n_warps, max(1LL, (T + p.min_units - 1) / p.min_units));
  const long long g = (long long)blockIdx.x * W + warp;
  if (g >= nwa) return;
  const long long wt0 = g * T / nwa, wt1 = (g + 1) * T / nwa;
  const int count = (int)(wt1 - wt0);
  const int start_b = seq_of_unit(wt0, pref, p.n_seq, spu);
  const uint64_t pol = l2_evict_first_policy();

  // raw query rows of a stream -> this warp's buffer (asynchronous copy)
  auto prefetch_queries = [&](int b, int h0) {
    const char *src = reinterpret_cast<const char *>(p.q + ((size_t)b * p.n_qh + h0) * D);
    for (int c = lane; c < C::kQBytes / 16; c += 32)
      cp_async_16(reinterpret_cast<char *>(qbuf) + c * 16, src + c * 16);
    cp_async_commit();
  };
  {
    int b = start_b;
    const UnitPos up = locate_unit(wt0, b, pref, spu);
    prefetch_queries(up.b, (up.si / p.n_sub) * GS * p.n_sub + (up.si % p.n_sub) * GS);
  }

  // ---- producer ---------------------------------------------------------------
  // Physical pages are fetched 32 units ahead, one per lane, so the issuing
  // lane never waits on the block table.  Only the last unit of a stream holds
  // the token the append grid writes in this step: the issuing lane waits for
  // that grid (programmatic dependent launch) before the first such unit and
  // requests everything else at once.
  int pcur = start_b;  // per-lane cursor of the page windows
  int win_base = 0;
  int win_page = lane < count ? page_of_unit(p, pref, spu, wt0 + lane, pcur) : -1;
  int nxt_page = -1;  // loaded once the first units are requested
  int ib = start_b;
  bool appended_visible = false;
  auto issue = [&](int i) {  // called by the whole warp, in unit order
    if (i - win_base >= 32) {
      win_base += 32;
      win_page = nxt_page;
      const int tn = win_base + 32 + lane;
      nxt_page = tn < count ? page_of_unit(p, pref, spu, wt0 + tn, pcur) : -1;
    }
    const int page = __shfl_sync(0xffffffffu, win_page, i - win_base);
    if (lane == 0) {
      const UnitPos up = locate_unit(wt0 + i, ib, pref, spu);
      if (up.u == up.units - 1 && !appended_visible) {
        pdl_wait_primary();
        appended_visible = true;
      }
      const int st = warp * C::kSW + i % C::kSW;
      svalid[i % C::kSW] = page >= 0;
      if (page >= 0) {
        const int row = (int)(((long long)page * p.n_kvh + up.si / p.n_sub) * p.page_size +
                              (up.u * kUnitRows) % p.page_size);
        uint8_t *dst = stages + (size_t)st * C::kStage;
        mbar_arrive_expect_tx(&bars[st], C::kStage);
#pragma unroll
        for (int r = 0; r < C::kRegions; ++r) {
          tma_load_2d(dst + r * C::kBox, &p.tmap_k, r * 64, row, &bars[st], pol);
          tma_load_2d(dst + C::kTile + r * C::kBox, &p.tmap_v, r * 64, row, &bars[st], pol);
        }
      } else {
        atomicOr(p.status, KVATTN_DEV_BAD_PAGE);
        mbar_arrive(&bars[st]);
      }
    }
  };
  int issued = 0;
  for (; issued < min(C::kSW, count); ++issued) issue(issued);
  if (32 + lane < count) nxt_page = page_of_unit(p, pref, spu, wt0 + 32 + lane, pcur);

  // ---- consumer ---------------------------------------------------------------
  const int hb = (GS == 4) ? 2 * (lane & 1) : 0;  // first head of this lane's columns
  bool aborted = false;
  int consumed = 0;
  int cb = start_b;
  long long t = wt0;
  while (t < wt1) {
    const UnitPos sp = locate_unit(t, cb, pref, spu);
    const long long F = sp.first, E = F + sp.units;
    const long long e = min(wt1, E);
    const int L = lens[sp.b];
    const int j = sp.si / p.n_sub, sub = sp.si % p.n_sub;
    const int h0 = j * GS * p.n_sub + sub * GS;
    const int sid = sp.b * spu + sp.si;

    uint32_t qb[C::kKSteps][2];
    float cr[D / 64], sr[D / 64];
    warp_query_angles<D>(p, turns, poss[sp.b], lane, cr, sr);  // while the rows land
    cp_async_wait_all();
    __syncwarp();
    warp_query_fragments<D, GS>(p, cr, sr, qbuf, lane, qb);
    __syncwarp();
    if (E < wt1) {  // the share continues: fetch the next stream's query rows
      int b = sp.b;
      const UnitPos nx = locate_unit(E, b, pref, spu);
      prefetch_queries(nx.b, (nx.si / p.n_sub) * GS * p.n_sub + (nx.si % p.n_sub) * GS);
    }
    float o[C::kKSteps][4];
#pragma unroll
    for (int dt = 0; dt < C::kKSteps; ++dt)
#pragma unroll
      for (int k = 0; k < 4; ++k) o[dt][k] = 0.f;
    float m[C::kHL], l[C::kHL];
#pragma unroll
    for (int h = 0; h < C::kHL; ++h) {
      m[h] = kNegInf;
      l[h] = 0.f;
    }

    for (long long tt = t; tt < e; ++tt) {
      const int i = (int)(tt - wt0);
      const int st = warp * C::kSW + i % C::kSW;
      bool ok = false;
      if (!aborted) {
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars[st], (uint32_t)((i / C::kSW) & 1)));
        if (!ok) {
          aborted = true;
          if (lane == 0) atomicOr(p.status, KVATTN_DEV_TIMEOUT);
        }
      }
      consumed = i + 1;
      const int tok0 = (int)(tt - F) * kUnitRows;
      if (ok && svalid[i % C::kSW]) {
        const int nrows = min(kUnitRows, L + 1 - tok0);
        uint8_t *Ks = stages + (size_t)st * C::kStage;
        uint8_t *Vs = Ks + C::kTile;
        const uint32_t kb = smem_addr(Ks), vb = smem_addr(Vs);
        if (nrows < kUnitRows) {
          // rows past the sequence end hold stale data: zero them in V so that
          // their zero weights cannot meet a NaN
          const int n16 = (kUnitRows - nrows) * C::kRegions * 8;
          for (int idx = lane; idx < n16; idx += 32) {
            const int row = nrows + idx / (C::kRegions * 8);
            const int c = idx % (C::kRegions * 8);
            *reinterpret_cast<uint4 *>(Vs + (c >> 3) * C::kBox + row * 128 + (c & 7) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          __syncwarp();
        }

        // S^T = K Qc^T
        float s[4] = {0.f, 0.f, 0.f, 0.f};
        {
          const int row = (lane & 7) + ((lane >> 3) & 1) * 8;
          const int csel = lane >> 4;
#pragma unroll
          for (int ks = 0; ks < C::kKSteps; ++ks) {
            uint32_t a[4];
            ldmatrix_x4(a, kb + (ks >> 2) * C::kBox + swz(row, ((ks & 3) << 1) + csel));
            mma_bf16_16816(s, a, qb[ks][0], qb[ks][1]);
          }
        }
        // full scores sc[token half][head slot] = hi column + lo column
        float sc[2][2];
        if constexpr (GS == 4) {
#pragma unroll
          for (int k = 0; k < 4; ++k) s[k] += __shfl_xor_sync(0xffffffffu, s[k], 2);
          sc[0][0] = s[0]; sc[0][1] = s[1]; sc[1][0] = s[2]; sc[1][1] = s[3];
        } else if constexpr (GS == 2) {
#pragma unroll
          for (int k = 0; k < 4; ++k) s[k] += __shfl_xor_sync(0xffffffffu, s[k], 1);
          sc[0][0] = s[0]; sc[0][1] = s[1]; sc[1][0] = s[2]; sc[1][1] = s[3];
        } else {
          sc[0][0] = s[0] + s[1]; sc[1][0] = s[2] + s[3];
          sc[0][1] = sc[1][1] = kNegInf;
        }
        const int tokr = lane >> 2;
        if (tokr >= nrows) sc[0][0] = sc[0][1] = kNegInf;
        if (tokr + 8 >= nrows) sc[1][0] = sc[1][1] = kNegInf;

        // online softmax (log2 units)
        float alpha[C::kHL], pw[2][C::kHL];
#pragma unroll
        for (int h = 0; h < C::kHL; ++h) {
          float mx = fmaxf(sc[0][h], sc[1][h]);
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          const float mn = fmaxf(m[h], mx);
          alpha[h] = (mn == kNegInf) ? 1.f : exp2f(m[h] - mn);
          m[h] = mn;
          pw[0][h] = (mn == kNegInf) ? 0.f : exp2f(sc[0][h] - mn);
          pw[1][h] = (mn == kNegInf) ? 0.f : exp2f(sc[1][h] - mn);
          l[h] = l[h] * alpha[h] + pw[0][h] + pw[1][h];
        }
        // P^T fragments: this lane's two columns at tokens r and r + 8, bf16
        // head or remainder of the weight, zero in padding columns
        uint32_t pr[2];
#pragma unroll
        for (int t2 = 0; t2 < 2; ++t2) {
          float x0, x1;
          if constexpr (GS == 4) {
            x0 = pw[t2][0];
            x1 = pw[t2][1];
            if (lane & 2) {
              x0 -= __bfloat162float(__float2bfloat16_rn(x0));
              x1 -= __bfloat162float(__float2bfloat16_rn(x1));
            }
          } else if constexpr (GS == 2) {
            x0 = pw[t2][0];
            x1 = pw[t2][1];
            if (lane & 1) {
              x0 -= __bfloat162float(__float2bfloat16_rn(x0));
              x1 -= __bfloat162float(__float2bfloat16_rn(x1));
            }
            if (lane & 2) x0 = x1 = 0.f;
          } else {
            x0 = pw[t2][0];
            x1 = x0 - __bfloat162float(__float2bfloat16_rn(x0));
            if (lane & 3) x0 = x1 = 0.f;
          }
          pr[t2] = pack_bf16(x0, x1);
        }
        const uint32_t b0 = movmatrix_trans(pr[0]);
        const uint32_t b1 = movmatrix_trans(pr[1]);
        // rescale the accumulators of this lane's columns
        const float a0 = alpha[0], a1 = alpha[C::kHL - 1];
#pragma unroll
        for (int dt = 0; dt < C::kKSteps; ++dt) {
          o[dt][0] *= a0; o[dt][1] *= a1; o[dt][2] *= a0; o[dt][3] *= a1;
        }
        // O^T += V^T P^T
        {
          const int row = (lane & 7) + (lane >> 4) * 8;
          const int csel = (lane >> 3) & 1;
#pragma unroll
          for (int dt = 0; dt < C::kKSteps; ++dt) {
            uint32_t a[4];
            ldmatrix_x4_trans(a, vb + (dt >> 2) * C::kBox + swz(row, ((dt & 3) << 1) + csel));
            mma_bf16_16816(o[dt], a, b0, b1);
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
    // add the remainder columns to the head columns; sum l over the tokens
#pragma unroll
    for (int dt = 0; dt < C::kKSteps; ++dt) {
      if constexpr (GS == 1) {
        o[dt][0] += o[dt][1];
        o[dt][2] += o[dt][3];
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k)
          o[dt][k] += __shfl_xor_sync(0xffffffffu, o[dt][k], GS == 4 ? 2 : 1);
      }
    }
#pragma unroll
    for (int h = 0; h < C::kHL; ++h) {
      l[h] += __shfl_xor_sync(0xffffffffu, l[h], 4);
      l[h] += __shfl_xor_sync(0xffffffffu, l[h], 8);
      l[h] += __shfl_xor_sync(0xffffffffu, l[h], 16);
    }
    // lanes holding final values: GS 4 -> lane % 4 in {0, 1} (heads hb, hb + 1);
    // GS 2 -> lane % 4 == 0 (heads 0, 1); GS 1 -> lane % 4 == 0 (head 0)
    const bool writer = (GS == 4) ? (lane & 2) == 0 : (lane & 3) == 0;
    const int dr = lane >> 2;
    __nv_bfloat16 *outp = p.out + ((size_t)sp.b * p.n_qh + h0) * D;
    if (F >= wt0 && E <= wt1) {
      if (writer) {
#pragma unroll
        for (int h = 0; h < C::kHL; ++h) {
          const float inv = l[h] > 0.f ? 1.f / l[h] : 0.f;
#pragma unroll
          for (int dt = 0; dt < C::kKSteps; ++dt) {
            outp[(hb + h) * D + dt * 16 + dr] = __float2bfloat16_rn(o[dt][h] * inv);
            outp[(hb + h) * D + dt * 16 + dr + 8] = __float2bfloat16_rn(o[dt][2 + h] * inv);
          }
        }
      }
    } else {
      // partial record of this warp's part: acc[GS][D] relative to 2^m, m, l
      float *rec = p.records + (size_t)(sid + g) * C::RS;
      if (writer) {
#pragma unroll
        for (int h = 0; h < C::kHL; ++h) {
#pragma unroll
          for (int dt = 0; dt < C::kKSteps; ++dt) {
            rec[(hb + h) * D + dt * 16 + dr] = o[dt][h];
            rec[(hb + h) * D + dt * 16 + dr + 8] = o[dt][2 + h];
          }
          if (dr == 0) {
            rec[GS * D + hb + h] = m[h];
            rec[GS * D + GS + hb + h] = l[h];
          }
        }
      }
    }
    t = e;
  }

  cp_async_wait_all();  // no query prefetch may land after the warp has left
  if (aborted && lane == 0) {
    for (int i = consumed; i < issued; ++i)
      (void)mbar_wait_bounded(&bars[warp * C::kSW + i % C::kSW], (uint32_t)((i / C::kSW) & 1));
  }
}

template <int D, int GS>
cudaError_t launch_decode_mma_t(const DecodeParams &p, int grid, cudaStream_t stream,
                                int *ctas_per_sm, bool launch) {
  using C = MmaCfg<D, GS>;
  auto kern = decode_mma_kernel<D, GS>;
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
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace kvattn
