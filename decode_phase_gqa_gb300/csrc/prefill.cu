// Paged chunked-prefill attention: each sequence b brings n_b >= 1 new tokens
// after the ctx_b tokens its pages already hold (a prompt, or the next chunk of
// one, or the k draft tokens of a speculative step to verify).  Two kernels on
// the caller's stream:
//
//  * append: the new keys and values go into slots ctx_b .. ctx_b + n_b - 1 of
//    the sequence's pages, the keys rotated by the same storage recipe as the
//    decode step's append (storage.cuh), new token i at RoPE position ctx_b + i;
//  * attention: new token i attends over the keys 0 .. ctx_b + i (its own
//    included, the later new ones masked), the causal attention of a prefill
//    ("LLM inference from smollm3.go", section "Prefill: the whole prompt at
//    once"; "Qwen3-8B inference engine from scratch in C++/CUDA", section
//    4.4.1: the blockwise softmax over key blocks, never the whole score
//    matrix).  With n_b = 1 it is the decode step.
//
// Attention kernel: a CTA takes 16 new tokens of one sequence and the 4 query
// heads of one group (a warp per head), so one staged K/V tile serves the 4
// heads (section 4.4.2 of the Qwen3-8B page: a group's KV is read once).
// Key tiles of 32 tokens are gathered page by page with 16-byte cp.async into
// a double-buffered, XOR-swizzled shared-memory ring; per tile a warp forms
// S = Q K^T (16 x 32, m16n8k16 bf16 MMAs, fp32), the online softmax of its 16
// rows in the log2 domain, and O += P V.  Query rows are rotated in fp32 and
// scaled by scale * log2(e) before they are rounded to bf16.
#include <algorithm>
#include <climits>
#include <cmath>
#include <type_traits>

#include "prefill_common.cuh"
#include "storage.cuh"

namespace kvattn {

namespace {

// The sequence of new-token row r: the last b < n_seq with seq_starts[b] <= r
// (the answer of a binary search when the starts ascend; a row the sequence
// does not hold is caught by the caller's seq_span check).  Called by a whole
// warp: each round its 32 lanes probe 32 evenly spaced starts of the range
// left and keep the piece after the last probe <= r, so 64 sequences take
// two rounds of loads instead of six dependent ones.
__device__ __forceinline__ int seq_of_row(const PrefillParams &p, int r, int lane) {
  int lo = 0, hi = p.n_seq;
  while (hi - lo > 1) {
    const int step = (hi - lo + 31) / 32;
    const int idx = lo + lane * step;
    const unsigned le = __ballot_sync(0xffffffffu, idx < hi && __ldg(p.seq_starts + idx) <= r);
    lo += le ? (31 - __clz(le)) * step : 0;
    hi = min(hi, lo + step);
  }
  return lo;
}

// Key tiles of the query tile starting at new token t0 (n_new new tokens after
// ctx cached ones), and the splits sharing them: S at most, each with at least
// kPfMinTiles tiles (the attention and merge kernels both use this).
__device__ __forceinline__ int query_tile_keys(int ctx, int n_new, int t0) {
  return ctx + min(n_new, t0 + kPfRows);
}
__device__ __forceinline__ int tile_splits(int n_tiles, int S) {
  return max(1, min(S, (n_tiles + kPfMinTiles - 1) / kPfMinTiles));
}
// the same for the short-chunk kernel's query tiles and 64-key stages
__device__ __forceinline__ int short_tile_keys(int ctx, int n_new) { return ctx + min(n_new, kPsTok); }
__device__ __forceinline__ int short_splits(int n_stages, int S) {
  return max(1, min(S, (n_stages + kPsMinTiles - 1) / kPsMinTiles));
}

// ---- append ------------------------------------------------------------------
// A warp per (new-token row, KV head); the CTA's four warps hold at most four
// tokens (one when n_kvh >= 4 divides evenly), and the RoPE angles of each token
// (an fp64 product reduced and rounded per pair, costly at this part's fp64
// rate) are formed once by the first warp holding it and shared: the row
// recipe is the decode step's (store_angle, rot_store, quant_row_warp), so the
// stored bits are the same.
template <int D, bool INT8>
__device__ __forceinline__ void stage_row_cs(const float2 *cs, bool use_rope, int lane, uint8_t *buf) {
  constexpr int PPL = D / 64;
  float xk[D / 32], xv[D / 32];
  const __nv_bfloat16 *raw = reinterpret_cast<const __nv_bfloat16 *>(buf);
#pragma unroll
  for (int k = 0; k < D / 32; ++k) {
    xk[k] = __bfloat162float(raw[row_elem<D>(lane, k)]);
    xv[k] = __bfloat162float(raw[D + row_elem<D>(lane, k)]);
  }
  __syncwarp();  // every lane has read the raw rows before the buffer is rewritten
  if (use_rope) {
#pragma unroll
    for (int k = 0; k < PPL; ++k) {
      const float2 a = cs[lane + 32 * k];
      rot_store(xk[k], xk[PPL + k], a.x, a.y, xk[k], xk[PPL + k]);
    }
  }
  if constexpr (INT8) {
    int8_t kc[D / 32], vc[D / 32];
    const float ksc = quant_row_warp<D>(xk, kc);
    const float vsc = quant_row_warp<D>(xv, vc);
    int8_t *kr = reinterpret_cast<int8_t *>(buf), *vr = kr + D;
#pragma unroll
    for (int k = 0; k < D / 32; ++k) {
      kr[row_elem<D>(lane, k)] = kc[k];
      vr[row_elem<D>(lane, k)] = vc[k];
    }
    if (lane == 0) {
      float *sc = reinterpret_cast<float *>(buf + 2 * D);
      sc[0] = ksc;
      sc[1] = vsc;
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

template <int D, bool INT8>
__global__ void __launch_bounds__(kPfThreads) prefill_append_kernel(const __grid_constant__ PrefillParams p) {
  __shared__ double inv_freq[64];
  __shared__ float4 table[sizeof(kSinCosStep) / 16];
  __shared__ __align__(16) uint8_t rowbuf[kPfWarps][4 * D];
  __shared__ float2 cs[kPfWarps][D / 2];  // (cos, sin) per pair, by the warp that formed them
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_launch_dependents();  // the attention grid may start at once
  if (tid < 64) inv_freq[tid] = p.inv_freq[tid];
  for (int i = tid; i < (int)(sizeof(kSinCosStep) / 16); i += kPfThreads) table[i] = kSinCosStep[i];
  const long long item0 = (long long)blockIdx.x * kPfWarps;
  const long long item = item0 + warp;  // (new-token row, KV head)
  const bool live = item < (long long)p.n_tok * p.n_kvh;
  const int r = live ? (int)(item / p.n_kvh) : 0, j = live ? (int)(item - (long long)r * p.n_kvh) : 0;
  // the new key and value rows are fetched (a 16-byte chunk a lane, held in
  // registers) while the row's sequence is found
  constexpr int CH = 2 * D / 16;  // 16-byte chunks of a row
  static_assert(2 * CH <= 32, "a chunk a lane");
  uint4 chunk = make_uint4(0u, 0u, 0u, 0u);
  if (live && lane < 2 * CH) {
    const uint4 *ks = reinterpret_cast<const uint4 *>(p.k_new + ((size_t)r * p.n_kvh + j) * D);
    const uint4 *vs = reinterpret_cast<const uint4 *>(p.v_new + ((size_t)r * p.n_kvh + j) * D);
    chunk = lane < CH ? ks[lane] : vs[lane - CH];
  }
  // the tcgen05 attention kernel's query rows (see below): the first four
  // heads of the group are fetched now too, so their latency overlaps the rest
  constexpr int QB = 4;                  // query heads fetched at once
  const int g = p.n_qh / p.n_kvh;
  __nv_bfloat16 qv[QB][2 * (D / 64)];    // element i = lane + 32 k and i + D / 2
  auto fetch_q = [&](int h_first) {
#pragma unroll
    for (int hh = 0; hh < QB; ++hh) {
      const bool in = live && h_first + hh < g;
      const __nv_bfloat16 *qs = p.q + ((size_t)r * p.n_qh + j * g + (in ? h_first + hh : 0)) * D;
#pragma unroll
      for (int k = 0; k < D / 64; ++k) {
        qv[hh][2 * k] = in ? qs[lane + 32 * k] : __float2bfloat16_rn(0.f);
        qv[hh][2 * k + 1] = in ? qs[lane + 32 * k + D / 2] : __float2bfloat16_rn(0.f);
      }
    }
  };
  if (p.tc_tiles) fetch_q(0);
  // (every test below depends on the token only, so all warps of a token agree)
  bool span_ok = false, ok = false;
  int lo = 0, slot = 0, page = 0;
  if (live) {
    lo = seq_of_row(p, r, lane);
    int start, n_new, ctx;
    // a row no valid sequence owns, or past the tokens the launch covers (the
    // attention kernel leaves those out too)
    if (!seq_span(p, lo, start, n_new, ctx) || r < start || r >= start + n_new ||
        r - start >= p.tiles_per_seq * p.tile_rows) {
      if (lane == 0 && j == 0) report(p, KVATTN_DEV_BAD_LEN);
    } else {
      span_ok = true;
      slot = ctx + (r - start);  // also the RoPE position
      page = __ldg(p.block_table + (size_t)lo * p.max_pages + (slot >> p.page_shift));
      if (page < 0 || page >= p.num_pages) {
        if (lane == 0 && j == 0) report(p, KVATTN_DEV_BAD_PAGE);
      } else {
        ok = true;
      }
    }
  }
  __shared__ int tok_slot[kPfWarps];  // RoPE position of each warp's token (-1: none)
  tok_slot[warp] = (span_ok && p.use_rope) ? slot : -1;
  __syncthreads();  // the tables and the positions
  // The angles of each token the CTA holds are formed once, into the slot of
  // the token's first warp (`owner`), by all the CTA's threads together: the
  // correctly rounded cos/sin of an fp64 angle is costly at this part's fp64
  // rate, and one warp doing a token's D/2 pairs alone is the CTA's longest
  // step.
  const int owner = (int)(max((long long)r * p.n_kvh, item0) - item0);
  for (int e = tid; e < kPfWarps * (D / 2); e += kPfThreads) {
    const int w = e / (D / 2), i = e - w * (D / 2);
    const long long it_w = item0 + w;
    const int own_w = (int)(max((it_w / p.n_kvh) * p.n_kvh, item0) - item0);  // first warp of w's token
    if (own_w != w || tok_slot[w] < 0) continue;
    float c, sn;
    store_angle_inl(tok_slot[w], inv_freq[i], table, c, sn);
    cs[w][i] = make_float2(c, sn);
  }
  __syncthreads();
  if (p.tc_tiles && span_ok) {
    // For the tcgen05 attention kernel the query rows of the KV head's group
    // are formed here, with the token's angles: rotated in fp32, scaled by
    // scale * log2(e), rounded to bf16, written to the output rows (which the
    // attention kernel reads by TMA and then overwrites with its result).
    // Four heads at a time, all loaded before any is stored.
#pragma unroll 1
    for (int h_first = 0; h_first < g; h_first += QB) {
      if (h_first > 0) fetch_q(h_first);
#pragma unroll
      for (int hh = 0; hh < QB; ++hh) {
        if (h_first + hh >= g) break;
        __nv_bfloat16 *qd = p.out + ((size_t)r * p.n_qh + j * g + h_first + hh) * D;
#pragma unroll
        for (int k = 0; k < D / 64; ++k) {
          const int i = lane + 32 * k;
          float lo = __bfloat162float(qv[hh][2 * k]), hi = __bfloat162float(qv[hh][2 * k + 1]);
          if (p.use_rope) {
            const float2 a = cs[owner][i];
            const float x = lo * a.x - hi * a.y, y = hi * a.x + lo * a.y;
            lo = x;
            hi = y;
          }
          qd[i] = __float2bfloat16_rn(lo * p.qscale);
          qd[i + D / 2] = __float2bfloat16_rn(hi * p.qscale);
        }
      }
    }
  }
  if (!ok) return;
  uint8_t *buf = rowbuf[warp];
  if (lane < 2 * CH) reinterpret_cast<uint4 *>(buf)[lane] = chunk;
  __syncwarp();
  stage_row_cs<D, INT8>(cs[owner], p.use_rope != 0, lane, buf);
  const size_t prow = ((size_t)page * p.n_kvh + j) * p.page_size + (slot & (p.page_size - 1));
  // the stored key row, then the value row (int8: codes, the two scales after)
  constexpr int RB = INT8 ? D : 2 * D, SCH = RB / 16;
  for (int c = lane; c < 2 * SCH; c += 32) {
    const uint4 x = reinterpret_cast<const uint4 *>(buf)[c];
    uint8_t *dst = static_cast<uint8_t *>(c < SCH ? p.k_pages : p.v_pages) + prow * RB;
    reinterpret_cast<uint4 *>(dst)[c < SCH ? c : c - SCH] = x;
  }
  if (INT8 && lane == 0) {
    const float *sc = reinterpret_cast<const float *>(buf + 2 * D);
    p.k_scales[prow] = sc[0];
    p.v_scales[prow] = sc[1];
  }
}

// ---- attention ---------------------------------------------------------------
template <int D, bool INT8>
struct PfCfg {
  static constexpr int kRowB = 2 * D;                        // bytes of a 16-bit row
  static constexpr int kQBytes = kPfWarps * kPfRows * kRowB;  // the warps' query rows
  static constexpr int kTile = kPfKeys * kRowB;              // one K or V tile (16-bit)
  static constexpr int kStage = 2 * kTile;                   // K then V
  // int8 cache: a stage's codes (K, V) and row scales (K, V) as copied
  static constexpr int kRaw = INT8 ? 2 * kPfKeys * D + 2 * kPfKeys * 4 : 0;
  static constexpr int kSmem = kQBytes + 2 * (kStage + kRaw) + 2 * kPfKeys * 4 + 64 * 8;
};

// The MMAs' 16-bit type: bf16 for the bf16 cache; f16 for the int8 cache,
// whose rows are dequantised (code * scale) into f16 tiles.
template <bool F16>
__device__ __forceinline__ uint32_t pack16(float lo, float hi) {
  if constexpr (F16) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
  } else {
    return pack_bf16(lo, hi);
  }
}
template <bool F16>
__device__ __forceinline__ uint16_t to16(float x) {
  if constexpr (F16) {
    __half v = __float2half_rn(x);
    return *reinterpret_cast<uint16_t *>(&v);
  } else {
    __nv_bfloat16 v = __float2bfloat16_rn(x);
    return *reinterpret_cast<uint16_t *>(&v);
  }
}
template <bool F16>
__device__ __forceinline__ void mma16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  if constexpr (F16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    mma_bf16_16816(d, a, b0, b1);
  }
}

// Byte offset of 16-byte chunk c of row r in a [rows][2 D] tile: the low three
// bits of the chunk index are XORed with the row's, so the 8 rows an ldmatrix
// reads at one chunk hit 8 different bank groups.
template <int D>
__device__ __forceinline__ uint32_t sw(int r, int c) {
  return (uint32_t)(r * 2 * D + (((c & ~7) | ((c ^ r) & 7)) << 4));
}

// 16-byte cp.async that copies `bytes` (16 or 0) and zero-fills the rest
__device__ __forceinline__ void cp_async_16_zfill(void *dst, const void *src, int bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_one() {
  asm volatile("cp.async.wait_group 1;" ::: "memory");
}

template <int D, bool INT8>
__global__ void __launch_bounds__(kPfThreads, 3) prefill_attn_kernel(const __grid_constant__ PrefillParams p) {
  using C = PfCfg<D, INT8>;
  constexpr int KS = D / 16;  // k-steps of Q K^T
  constexpr int ND = D / 8;   // n-tiles of O
  constexpr int CH = D / 8;   // 16-byte chunks of a row
  const float kFloor = -1e30f;  // initial running maximum, below any score
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t *qs = smem;
  uint8_t *stages = smem + C::kQBytes;
  uint8_t *raws = stages + 2 * C::kStage;  // int8: [2][codes K, codes V, scales K, scales V]
  int *rvalid = reinterpret_cast<int *>(raws + 2 * C::kRaw);  // [2][kPfKeys]
  float2 *turns = reinterpret_cast<float2 *>(rvalid + 2 * kPfKeys);  // [64]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // CTA x: head group x % G, then sequence, then query tile from the last:
  // the latest tiles of every sequence and group (the most keys) are placed
  // first, so the longest CTAs do not start last
  const int G = p.n_qh / kPfWarps;
  const int grp = (int)(blockIdx.x % G), rest = (int)(blockIdx.x / G);
  const int b = rest % p.n_seq, qt = p.tiles_per_seq - 1 - rest / p.n_seq;
  const int g = p.n_qh / p.n_kvh;
  const int j = grp / (g / kPfWarps);
  const int h = j * g + (grp % (g / kPfWarps)) * kPfWarps + warp;  // this warp's head
  // Launched as the append kernel's programmatic dependent: the queries are
  // formed while the append runs, and every thread waits for the append grid
  // before the first key tile (or before it leaves).
  int start, n_new, ctx;
  if (!seq_span(p, b, start, n_new, ctx)) {
    if (qt == 0 && grp == 0 && tid == 0) report(p, KVATTN_DEV_BAD_LEN);
    pdl_wait_primary();
    return;
  }
  // more new tokens than the grid's tiles cover (a bound the caller gave)
  if (qt == 0 && grp == 0 && tid == 0 && n_new > p.tiles_per_seq * kPfRows)
    report(p, KVATTN_DEV_BAD_LEN);
  const int t0 = qt * kPfRows;
  if (t0 >= n_new) {
    pdl_wait_primary();
    return;
  }
  // keys the CTA's last valid row sees: 0 .. ctx + min(n_new, t0 + 16) - 1, in
  // tiles; split z of the query tile takes a contiguous range of them (a split
  // past the query tile's count has nothing to do)
  const int n_keys = query_tile_keys(ctx, n_new, t0);
  const int n_tiles = (n_keys + kPfKeys - 1) / kPfKeys;
  const int z = blockIdx.z, nz = tile_splits(n_tiles, p.n_splits);
  if (z >= nz) {
    pdl_wait_primary();
    return;
  }
  const int per = (n_tiles + nz - 1) / nz;
  const int kt_begin = z * per, kt_end = min(n_tiles, kt_begin + per);
  if (tid < 64) turns[tid] = p.turns[tid];
  __syncthreads();

  // ---- the warp's 16 query rows: rotated in fp32, scaled, rounded to bf16 ----
  // lane: row lane / 2, blocks of 8 dimension pairs (i, i + D / 2) from
  // i0 = 8 (lane % 2 + 2 m), m < NB: all loads (16 bytes each) issued at once
  uint8_t *qw = qs + warp * kPfRows * C::kRowB;
  {
    constexpr int NB = D / 32;
    const int r = lane >> 1;
    const bool has = t0 + r < n_new;
    const __nv_bfloat16 *qr = p.q + ((size_t)(start + t0 + (has ? r : 0)) * p.n_qh + h) * D;
    uint4 qlo[NB], qhi[NB];
#pragma unroll
    for (int m = 0; m < NB; ++m) {
      const int i0 = 8 * ((lane & 1) + 2 * m);
      qlo[m] = has ? __ldg(reinterpret_cast<const uint4 *>(qr + i0)) : make_uint4(0u, 0u, 0u, 0u);
      qhi[m] = has ? __ldg(reinterpret_cast<const uint4 *>(qr + i0 + D / 2)) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int m = 0; m < NB; ++m) {
      const int i0 = 8 * ((lane & 1) + 2 * m);
      const __nv_bfloat16 *lo16 = reinterpret_cast<const __nv_bfloat16 *>(&qlo[m]);
      const __nv_bfloat16 *hi16 = reinterpret_cast<const __nv_bfloat16 *>(&qhi[m]);
      uint16_t olo[8], ohi[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        float lo = __bfloat162float(lo16[k]), hi = __bfloat162float(hi16[k]);
        if (p.use_rope && has) {
          float sn, cs;
          sincospif(2.f * frac_turns(ctx + t0 + r, turns[i0 + k]), &sn, &cs);
          const float a = lo * cs - hi * sn, bb = hi * cs + lo * sn;
          lo = a;
          hi = bb;
        }
        olo[k] = to16<INT8>(lo * p.qscale);
        ohi[k] = to16<INT8>(hi * p.qscale);
      }
      *reinterpret_cast<uint4 *>(qw + sw<D>(r, i0 / 8)) = *reinterpret_cast<const uint4 *>(olo);
      *reinterpret_cast<uint4 *>(qw + sw<D>(r, (i0 + D / 2) / 8)) = *reinterpret_cast<const uint4 *>(ohi);
    }
  }
  __syncwarp();
  uint32_t qf[KS][4];  // A fragments: rows g, g + 8; k 2t.., 2t + 8..
#pragma unroll
  for (int ks = 0; ks < KS; ++ks)
    ldmatrix_x4(qf[ks], smem_addr(qw) + sw<D>((lane & 7) + ((lane >> 3) & 1) * 8, 2 * ks + (lane >> 4)));

  // ---- key tiles ----------------------------------------------------------------
  // pool row of key token tok, or -1 (past the keys, or an out-of-range page)
  auto pool_row = [&](int tok, bool rep) -> long long {
    if (tok >= n_keys) return -1;
    const int page = __ldg(p.block_table + (size_t)b * p.max_pages + (tok >> p.page_shift));
    if (page < 0 || page >= p.num_pages) {
      if (rep) report(p, KVATTN_DEV_BAD_PAGE);
      return -1;
    }
    return ((long long)page * p.n_kvh + j) * p.page_size + (tok & (p.page_size - 1));
  };
  auto load_tile = [&](int kt, int s) {
    constexpr int RB = INT8 ? D : 2 * D;  // bytes of a cached row
    constexpr int RCH = RB / 16;
    // bf16: straight into the swizzled tiles; int8: the codes into the raw area
    uint8_t *Kd = INT8 ? raws + s * C::kRaw : stages + s * C::kStage;
    uint8_t *Vd = INT8 ? Kd + kPfKeys * D : Kd + C::kTile;
    for (int idx = tid; idx < kPfKeys * RCH; idx += kPfThreads) {
      const int r = idx / RCH, c = idx % RCH;
      const long long prow = pool_row(kt * kPfKeys + r, c == 0);
      const uint8_t *srck = static_cast<const uint8_t *>(p.k_pages);
      const uint8_t *srcv = static_cast<const uint8_t *>(p.v_pages);
      if (prow >= 0) {
        srck += prow * RB + c * 16;
        srcv += prow * RB + c * 16;
      }
      const uint32_t off = INT8 ? (uint32_t)(r * D + c * 16) : sw<D>(r, c);
      cp_async_16_zfill(Kd + off, srck, prow >= 0 ? 16 : 0);
      cp_async_16_zfill(Vd + off, srcv, prow >= 0 ? 16 : 0);
      if (c == 0) rvalid[s * kPfKeys + r] = prow >= 0;
    }
    if constexpr (INT8) {
      // row scales: each 16-key half of the tile lies in one page (64 bytes
      // of K scales, 64 of V); 16-byte copies, zero-filled past the keys
      if (tid < 4 * (kPfKeys / 16) * 2) {
        const int half = tid >> 3, v = (tid >> 2) & 1, part = tid & 3;
        const long long prow = pool_row(kt * kPfKeys + 16 * half, false);
        const float *src = v ? p.v_scales : p.k_scales;
        if (prow >= 0) src += prow + 4 * part;
        float *dst = reinterpret_cast<float *>(Kd + 2 * kPfKeys * D) + v * kPfKeys + 16 * half + 4 * part;
        cp_async_16_zfill(dst, src, prow >= 0 ? 16 : 0);
      }
    }
    cp_async_commit();
  };

  float o[ND][4];
#pragma unroll
  for (int nd = 0; nd < ND; ++nd)
#pragma unroll
    for (int k = 0; k < 4; ++k) o[nd][k] = 0.f;
  float m[2] = {kFloor, kFloor}, l[2] = {0.f, 0.f};
  float dmo[2] = {kFloor, kFloor};  // int8: the value weights' running maximum, less m
  // absolute positions of this lane's rows g and g + 8
  const int qpos[2] = {ctx + t0 + (lane >> 2), ctx + t0 + (lane >> 2) + 8};

  // this CTA's key tiles: kt_begin .. kt_end - 1 (split z of nz)
  pdl_wait_primary();  // the appended rows are complete and visible
  if (kt_begin < kt_end)
    load_tile(kt_begin, 0);
  else
    cp_async_commit();
  for (int it = 0, kt = kt_begin; kt < kt_end; ++it, ++kt) {
    if (kt + 1 < kt_end)
      load_tile(kt + 1, (it + 1) & 1);
    else
      cp_async_commit();  // (an empty group: the wait below still means tile kt)
    cp_async_wait_one();
    __syncthreads();
    const uint8_t *Ks = stages + (it & 1) * C::kStage, *Vs = Ks + C::kTile;
    const int *rv = rvalid + (it & 1) * kPfKeys;
    if constexpr (INT8) {
      // the stage's codes -> exact f16 tiles (rows not to be read: zero); the
      // row scales enter the scores and the value weights below, so no f16
      // product of a code and a scale can overflow or lose range
      const int8_t *raw = reinterpret_cast<const int8_t *>(raws + (it & 1) * C::kRaw);
      for (int idx = tid; idx < 2 * kPfKeys * CH; idx += kPfThreads) {
        const int v = idx / (kPfKeys * CH), rest = idx - v * kPfKeys * CH;
        const int r = rest / CH, c = rest % CH;
        const float sc = rv[r] ? 1.f : 0.f;
        const uint2 w = *reinterpret_cast<const uint2 *>(raw + v * kPfKeys * D + r * D + c * 8);
        const int8_t *e = reinterpret_cast<const int8_t *>(&w);
        uint4 o4;
        o4.x = pack16<true>(e[0] * sc, e[1] * sc);
        o4.y = pack16<true>(e[2] * sc, e[3] * sc);
        o4.z = pack16<true>(e[4] * sc, e[5] * sc);
        o4.w = pack16<true>(e[6] * sc, e[7] * sc);
        *reinterpret_cast<uint4 *>(const_cast<uint8_t *>(v ? Vs : Ks) + sw<D>(r, c)) = o4;
      }
      __syncthreads();
    }
    const uint32_t kb = smem_addr(Ks), vb = smem_addr(Vs);

    // S = Q K^T over the tile's keys, n-tiles of 8 keys
    float s[kPfNT][4];
#pragma unroll
    for (int nt = 0; nt < kPfNT; ++nt)
#pragma unroll
      for (int k = 0; k < 4; ++k) s[nt][k] = 0.f;
#pragma unroll
    for (int nt = 0; nt < kPfNT; nt += 2) {
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        // matrices: keys nt*8.. at chunks 2ks, 2ks+1, then keys (nt+1)*8.. at the same
        uint32_t kf[4];
        const int mi = lane >> 3;
        ldmatrix_x4(kf, kb + sw<D>((nt + (mi >> 1)) * 8 + (lane & 7), 2 * ks + (mi & 1)));
        mma16<INT8>(s[nt], qf[ks], kf[0], kf[1]);
        mma16<INT8>(s[nt + 1], qf[ks], kf[2], kf[3]);
      }
    }
    // causal and page masks, running maxima of rows g and g + 8
    const int key0 = kt * kPfKeys;
    // int8: the raw dot products times the key rows' scales; the value weights
    // are 2^(S - m + log2 vs - dmo) with their own running maximum m + dmo, so
    // P vs fits f16 whatever the scales, and log2 vs is added to a number near
    // zero, which fp32 keeps whatever the scores' size (the decode kernel's
    // scheme)
    const float *scl = INT8 ? reinterpret_cast<const float *>(raws + (it & 1) * C::kRaw + 2 * kPfKeys * D)
                            : nullptr;
    float mx[2] = {-INFINITY, -INFINITY};
    float xv[kPfNT][4];  // int8: log2 vs, then the value-weight exponents
#pragma unroll
    for (int nt = 0; nt < kPfNT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int kr = nt * 8 + 2 * (lane & 3) + (e & 1);
        const bool ok = key0 + kr <= qpos[e >> 1] && rv[kr] != 0;
        if constexpr (INT8) {
          s[nt][e] = ok ? s[nt][e] * scl[kr] : -INFINITY;
          xv[nt][e] = ok ? lg2_approx(scl[kPfKeys + kr]) : -INFINITY;
        } else {
          s[nt][e] = ok ? s[nt][e] : -INFINITY;
        }
        mx[e >> 1] = fmaxf(mx[e >> 1], s[nt][e]);
      }
    float alpha[2], alpha_o[2];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xffffffffu, mx[rr], 1));
      mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xffffffffu, mx[rr], 2));
      const float mn = fmaxf(m[rr], mx[rr]);
      alpha[rr] = ex2_approx(m[rr] - mn);
      if constexpr (INT8) dmo[rr] -= mn - m[rr];  // the same absolute reference
      m[rr] = mn;
      l[rr] *= alpha[rr];
      alpha_o[rr] = alpha[rr];
    }
    if constexpr (INT8) {
      float mxo[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int nt = 0; nt < kPfNT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          xv[nt][e] += s[nt][e] - m[e >> 1];
          mxo[e >> 1] = fmaxf(mxo[e >> 1], xv[nt][e]);
        }
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        mxo[rr] = fmaxf(mxo[rr], __shfl_xor_sync(0xffffffffu, mxo[rr], 1));
        mxo[rr] = fmaxf(mxo[rr], __shfl_xor_sync(0xffffffffu, mxo[rr], 2));
        const float don = fmaxf(dmo[rr], mxo[rr]);
        alpha_o[rr] = ex2_approx(dmo[rr] - don);
        dmo[rr] = don;
      }
    }
#pragma unroll
    for (int nt = 0; nt < kPfNT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        s[nt][e] = ex2_approx(s[nt][e] - m[e >> 1]);
        l[e >> 1] += s[nt][e];
        if constexpr (INT8) s[nt][e] = ex2_approx(xv[nt][e] - dmo[e >> 1]);  // the value weight
      }
#pragma unroll
    for (int nd = 0; nd < ND; ++nd) {
      o[nd][0] *= alpha_o[0];
      o[nd][1] *= alpha_o[0];
      o[nd][2] *= alpha_o[1];
      o[nd][3] *= alpha_o[1];
    }
    // O += P V: P's accumulator layout is the next MMA's A layout, keys
    // 16 kk .. 16 kk + 15 from n-tiles 2 kk, 2 kk + 1
#pragma unroll
    for (int kk = 0; kk < kPfKK; ++kk) {
      const uint32_t a[4] = {pack16<INT8>(s[2 * kk][0], s[2 * kk][1]),
                             pack16<INT8>(s[2 * kk][2], s[2 * kk][3]),
                             pack16<INT8>(s[2 * kk + 1][0], s[2 * kk + 1][1]),
                             pack16<INT8>(s[2 * kk + 1][2], s[2 * kk + 1][3])};
#pragma unroll
      for (int nd = 0; nd < ND; nd += 2) {
        // matrices: keys 16kk..+7 and 16kk+8..+15 at chunk nd, then at chunk nd+1
        uint32_t vf[4];
        ldmatrix_x4_trans(vf, vb + sw<D>(16 * kk + (lane & 7) + ((lane >> 3) & 1) * 8, nd + (lane >> 4)));
        mma16<INT8>(o[nd], a, vf[0], vf[1]);
        mma16<INT8>(o[nd + 1], a, vf[2], vf[3]);
      }
    }
    __syncthreads();  // the stage is rewritten two tiles on
  }
  cp_async_wait_all();

  // ---- rows g and g + 8 of head h: O / l, rounded to bf16 ----------------------
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    l[rr] += __shfl_xor_sync(0xffffffffu, l[rr], 1);
    l[rr] += __shfl_xor_sync(0xffffffffu, l[rr], 2);
    if constexpr (INT8) {  // o is relative to 2^(m + dmo): bring it to 2^m
      const float f = ex2_approx(dmo[rr]);
#pragma unroll
      for (int nd = 0; nd < ND; ++nd) {
        o[nd][2 * rr] *= f;
        o[nd][2 * rr + 1] *= f;
      }
    }
  }
  if (p.n_splits > 1) {  // a partial state per row, merged by prefill_merge_kernel
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int t = t0 + (lane >> 2) + 8 * rr;
      if (t >= n_new) continue;
      float *rec = p.part + (((size_t)z * p.n_tok + start + t) * p.n_qh + h) * (D + 2);
#pragma unroll
      for (int nd = 0; nd < ND; ++nd)
        *reinterpret_cast<float2 *>(rec + 8 * nd + 2 * (lane & 3)) =
            make_float2(o[nd][2 * rr], o[nd][2 * rr + 1]);
      if ((lane & 3) == 0) *reinterpret_cast<float2 *>(rec + D) = make_float2(m[rr], l[rr]);
    }
    return;
  }
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    const int t = t0 + (lane >> 2) + 8 * rr;
    if (t >= n_new) continue;
    const float f = l[rr] > 0.f ? 1.f / l[rr] : 0.f;  // no visible key: a zero row
    __nv_bfloat162 *dst = reinterpret_cast<__nv_bfloat162 *>(
        p.out + ((size_t)(start + t) * p.n_qh + h) * D + 2 * (lane & 3));
#pragma unroll
    for (int nd = 0; nd < ND; ++nd)
      dst[4 * nd] = __floats2bfloat162_rn(o[nd][2 * rr] * f, o[nd][2 * rr + 1] * f);
  }
}

// ---- short chunks: at most 4 new tokens a sequence ------------------------------
// The 16 MMA rows are the 4 new tokens x the 4 query heads of a group (row
// 4 t + i: token t, head i), so no row is padding when the chunk is a
// speculative step's drafts.  A 64-key stage is split among the 4 warps (16
// keys each); each warp streams its own 16 keys of every stage (one page)
// through a private ring of stages that TMA tensor copies fill ([16 rows]
// boxes of the pool, 128- or 64-byte swizzle, the decode kernel's views),
// each stage with its own barrier, so warps stream independently with no CTA
// barrier per stage.  Each warp keeps its own online-softmax state of all 16
// rows; the four states are merged in shared memory at the end.
template <int D, bool INT8>
struct PsCfg {
  static constexpr int kRowB = 2 * D;                 // a query row (16-bit)
  static constexpr int kQBytes = 16 * kRowB;
  static constexpr int kCacheRowB = INT8 ? D : 2 * D;  // a cached row
  static constexpr int kBoxB = kCacheRowB < 128 ? kCacheRowB : 128;  // bytes of a box row
  static constexpr int kRegions = kCacheRowB / kBoxB;  // boxes a 16-row tile
  static constexpr int kBox = kPsWarpKeys * kBoxB;
  static constexpr int kTile = kRegions * kBox;        // a warp's K (or V) rows of a stage
  static constexpr int kStage = 2 * kTile;             // K then V
  // stages of a warp's ring: the int8 slices are half the bytes, so twice as
  // many fit the same shared memory (3 CTAs an SM either way)
  static constexpr int kStages = INT8 ? 2 * kPsStages : kPsStages;
  static constexpr int kRing = kStages * kStage;       // a warp's
  // after 1024 bytes of alignment slack: the rings, the query rows, the int8
  // row scales [warp][stage][K 16, V 16], the stage barriers, the RoPE turns
  static constexpr int kQOff = kPfWarps * kRing;
  static constexpr int kScaleOff = kQOff + kQBytes;
  static constexpr int kBarOff = kScaleOff + (INT8 ? kPfWarps * kStages * 2 * kPsWarpKeys * 4 : 0);
  static constexpr int kTurnsOff = kBarOff + kPfWarps * kStages * 8;
  static constexpr int kSmem = 1024 + kTurnsOff + 64 * 8;
  static_assert(kBox % 1024 == 0 || (kBoxB == 64 && kBox % 512 == 0), "swizzled boxes need alignment");
  // the end-of-kernel merge borrows the rings: [4 warps][16 rows][D] + (m, l)
  static_assert(kPfWarps * 16 * (D + 2) * 4 <= kPfWarps * kRing, "merge buffer");
};

// The short kernel's parameters: the call's, and the pools' TMA views
struct PsParams {
  PrefillParams p;
  CUtensorMap tmap_k, tmap_v;
};

// Byte offset of 16-byte chunk c of row r in a bf16 K or V tile as the TMA
// writes it: boxes of [16 rows][128 bytes] one after another, the chunk index
// XORed with the row's low three bits (128-byte swizzle)
template <int D>
__device__ __forceinline__ uint32_t tile_sw(int r, int c) {
  return (uint32_t)((c >> 3) * (kPsWarpKeys * 128) + r * 128 + (((c ^ r) & 7) << 4));
}

// Position of 16-byte chunk c of code row r in a staged int8 slice [16][D]:
// XOR-permuted so that the 8 rows an ldmatrix reads at one chunk fall in 8
// different bank groups (rows of 128 bytes: with r mod 8; of 64 bytes, two to
// 128 bytes: with (r / 2) mod 4)
template <int D>
__device__ __forceinline__ int cidx8(int r, int c) {
  return D == 128 ? (c ^ (r & 7)) : (c ^ ((r >> 1) & 3));
}

template <int N>
__device__ __forceinline__ void cp_async_wait_n() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <int D, bool INT8>
__global__ void __launch_bounds__(kPfThreads, 3) prefill_short_kernel(const __grid_constant__ PsParams sp) {
  using C = PsCfg<D, INT8>;
  const PrefillParams &p = sp.p;
  constexpr int KS = D / 16;
  constexpr int ND = D / 8;
  const float kFloor = -1e30f;
  const float kLazy = 8.f;  // log2 headroom of the lazy softmax references
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint8_t *rings = smem;
  uint8_t *qs = smem + C::kQOff;
  float2 *turns = reinterpret_cast<float2 *>(smem + C::kTurnsOff);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = p.n_qh / kPfWarps;  // head quads
  const int grp = (int)(blockIdx.x % G), b = (int)(blockIdx.x / G);
  const int g = p.n_qh / p.n_kvh;
  const int j = grp / (g / kPfWarps);
  const int h0 = j * g + (grp % (g / kPfWarps)) * kPfWarps;  // the quad's first head
  // (the frequencies first: their load from the parameters overlaps the
  // sequence's)
  if (tid < 64) turns[tid] = p.turns[tid];
  int start, n_new, ctx;
  // Launched as the append kernel's programmatic dependent: the cached keys
  // (slots below ctx) are read while the append runs; a warp waits for the
  // append grid before its first slice that holds new slots, and every
  // working thread waits before it leaves, so the grid ends after the
  // append's.  CTAs with nothing to do leave at once (the first CTA waits
  // all the same, so that the grid cannot end before the append's).
  const bool first_cta = blockIdx.x == 0 && blockIdx.z == 0;
  if (!seq_span(p, b, start, n_new, ctx)) {
    if (grp == 0 && blockIdx.z == 0 && tid == 0) report(p, KVATTN_DEV_BAD_LEN);
    if (first_cta) pdl_wait_primary();
    return;
  }
  if (grp == 0 && blockIdx.z == 0 && tid == 0 && n_new > kPsTok) report(p, KVATTN_DEV_BAD_LEN);
  const int n_keys = short_tile_keys(ctx, n_new);
  const int n_tiles = (n_keys + kPsKeys - 1) / kPsKeys;
  const int z = blockIdx.z, nz = short_splits(n_tiles, p.n_splits);
  if (n_new <= 0 || z >= nz) {
    if (first_cta) pdl_wait_primary();
    return;
  }
  // Split z takes stages [B(z), B(z + 1)), B(z) = n (1 - r^z) / (1 - r^nz)
  // rounded, r = 3/4: each split a quarter shorter than the one before.  The
  // grid is placed split by split, so the CTAs placed last, while the GPU
  // drains, are the short ones (equal splits left a tail of whole splits
  // started late).  A split may come out empty: it leaves an empty state.
  const auto bound = [&](int zz) -> int {
    if (zz >= nz) return n_tiles;
    float pz = 1.f, pn = 1.f;
    for (int k = 0; k < nz; ++k) {
      if (k < zz) pz *= 0.75f;
      pn *= 0.75f;
    }
    return (int)((float)n_tiles * ((1.f - pz) / (1.f - pn)) + 0.5f);
  };
  const int kt_begin = bound(z), kt_end = bound(z + 1);

  const int wk = warp * kPsWarpKeys;  // the warp's keys within a stage
  uint8_t *ring = rings + warp * C::kRing;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kBarOff) + warp * C::kStages;
  float *wscl = reinterpret_cast<float *>(smem + C::kScaleOff) + warp * C::kStages * 2 * kPsWarpKeys;
  if (lane == 0) {
    for (int s = 0; s < C::kStages; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
    prefetch_tensormap(&sp.tmap_k);
    prefetch_tensormap(&sp.tmap_v);
  }
  __syncthreads();  // (the turns; the barriers are the warp's own)
  const uint64_t pol = l2_evict_first_policy();
  uint32_t bad = 0;  // bit s: stage s's keys lie in an out-of-range page (nothing copied)
  bool appended = false;  // the append grid is complete and its rows visible
  // Block-table entries of the warp's stages, 32 at a time: lane i holds the
  // page of stage win_base + i, so a stage's copies never wait on a table
  // load (the table is no output of the append grid)
  const int *bt_row = p.block_table + (size_t)b * p.max_pages;
  auto stage_page = [&](int kt) {
    const int key = kt * kPsKeys + wk;
    return (kt < kt_end && key < n_keys) ? __ldg(bt_row + (key >> p.page_shift)) : -1;
  };
  int win_base = kt_begin;
  int win_page = stage_page(kt_begin + lane);
  // The warp's 16 keys of stage kt (one page: pages hold 16 keys or more)
  // into ring slot s: TMA boxes of K and V (the 16 rows of the page slots;
  // rows past the keys come as the pool holds them and are masked, bf16 V
  // rows zeroed), the int8 row scales by two bulk copies, all on the slot's
  // barrier.  Called for kt = kt_begin, kt_begin + 1, ... in order, by the
  // whole warp.
  auto load_part = [&](int kt, int s) {
    const int key = kt * kPsKeys + wk;
    if (kt - win_base >= 32) {
      win_base += 32;
      win_page = stage_page(win_base + lane);
    }
    const int page = __shfl_sync(0xffffffffu, win_page, kt - win_base);
    if (!appended && key + kPsWarpKeys > ctx) {
      pdl_wait_primary();
      appended = true;
    }
    int row = -1;
    if (key < n_keys) {
      if (page >= 0 && page < p.num_pages)
        row = (page * p.n_kvh + j) * p.page_size + (key & (p.page_size - 1));
      else if (lane == 0)
        report(p, KVATTN_DEV_BAD_PAGE);
    }
    bad = row >= 0 ? bad & ~(1u << s) : bad | (1u << s);
    __syncwarp();  // every lane is done with the slot (and its bf16 zeroing)
    if (lane == 0) {
      if (row >= 0) {
        fence_proxy_async_smem();  // those generic accesses before the copy's writes
        uint8_t *dst = ring + s * C::kStage;
        mbar_arrive_expect_tx(&bars[s], C::kStage + (INT8 ? 2 * kPsWarpKeys * 4 : 0));
        if constexpr (INT8) {
          // the 16 rows' key and value scales: 64 bytes each, 64-byte aligned
          // (the warp's 16 keys start a 16-row block of the page)
          float *ws = wscl + s * 2 * kPsWarpKeys;
          bulk_g2s(ws, p.k_scales + row, kPsWarpKeys * 4, &bars[s], pol);
          bulk_g2s(ws + kPsWarpKeys, p.v_scales + row, kPsWarpKeys * 4, &bars[s], pol);
        }
#pragma unroll
        for (int r = 0; r < C::kRegions; ++r) {
          const int x = r * C::kBoxB / (INT8 ? 1 : 2);  // element column of box r
          tma_load_2d(dst + r * C::kBox, &sp.tmap_k, x, row, &bars[s], pol);
          tma_load_2d(dst + C::kTile + r * C::kBox, &sp.tmap_v, x, row, &bars[s], pol);
        }
      } else {
        mbar_arrive(&bars[s]);
      }
    }
  };
  // The 16 query rows (token r / 4, head h0 + r % 4), rotated and scaled: warp
  // t takes token t, a thread PP dimension pairs (i, i + D / 2) from
  // i0 = PP lane for all four heads (one angle serves the four).  The loads
  // go out before the first stages' copies and the angles are formed while
  // they are in flight (the latency of a row of dependent two-byte loads
  // dominated the CTA's set-up).
  constexpr int PP = D / 64;
  static_assert(16 * (D / 2) == 4 * PP * kPfThreads, "a thread's pairs");
  using QVec = typename std::conditional<PP == 2, uint32_t, uint16_t>::type;
  const int qt = warp, qi0 = lane * PP;
  const bool qlive = qt < n_new;
  QVec qlo[4], qhi[4];
  {
    const __nv_bfloat16 *qr = p.q + ((size_t)(start + (qlive ? qt : 0)) * p.n_qh + h0) * D + qi0;
#pragma unroll
    for (int hh = 0; hh < 4; ++hh) {
      qlo[hh] = qlive ? __ldg(reinterpret_cast<const QVec *>(qr + hh * D)) : QVec(0);
      qhi[hh] = qlive ? __ldg(reinterpret_cast<const QVec *>(qr + hh * D + D / 2)) : QVec(0);
    }
  }
  float qcs[PP], qsn[PP];
#pragma unroll
  for (int k = 0; k < PP; ++k) {
    qcs[k] = 1.f;
    qsn[k] = 0.f;
    if (p.use_rope && qlive) sincospif(2.f * frac_turns(ctx + qt, turns[qi0 + k]), &qsn[k], &qcs[k]);
  }
  // the first stages go out before the queries are formed
  int issued = 0;
  for (; issued < C::kStages - 1 && kt_begin + issued < kt_end; ++issued) load_part(kt_begin + issued, issued);

#pragma unroll
  for (int hh = 0; hh < 4; ++hh) {
    const __nv_bfloat16 *lo16 = reinterpret_cast<const __nv_bfloat16 *>(&qlo[hh]);
    const __nv_bfloat16 *hi16 = reinterpret_cast<const __nv_bfloat16 *>(&qhi[hh]);
    uint16_t olo[PP], ohi[PP];
#pragma unroll
    for (int k = 0; k < PP; ++k) {
      float lo = __bfloat162float(lo16[k]), hi = __bfloat162float(hi16[k]);
      if (p.use_rope && qlive) {
        const float a = lo * qcs[k] - hi * qsn[k], bb = hi * qcs[k] + lo * qsn[k];
        lo = a;
        hi = bb;
      }
      olo[k] = to16<INT8>(lo * p.qscale);
      ohi[k] = to16<INT8>(hi * p.qscale);
    }
    const int r = 4 * qt + hh;
    *reinterpret_cast<QVec *>(qs + sw<D>(r, qi0 / 8) + (qi0 % 8) * 2) = *reinterpret_cast<const QVec *>(olo);
    *reinterpret_cast<QVec *>(qs + sw<D>(r, (qi0 + D / 2) / 8) + ((qi0 + D / 2) % 8) * 2) =
        *reinterpret_cast<const QVec *>(ohi);
  }
  __syncthreads();
  uint32_t qf[KS][4];
  if constexpr (INT8) {
    // the k order of the key codes' fragments (below): MMA columns 2t, 2t + 1
    // of k-step ks are dimensions 16 ks + 4t, + 1, columns 2t + 8, 2t + 9 are
    // 16 ks + 4t + 2, + 3 (t = lane % 4): one 8-byte load per row
    const int t4 = lane & 3, g8 = lane >> 2;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const uint32_t off = (uint32_t)((t4 & 1) * 8);
      const uint2 r0 = *reinterpret_cast<const uint2 *>(qs + sw<D>(g8, 2 * ks + (t4 >> 1)) + off);
      const uint2 r1 = *reinterpret_cast<const uint2 *>(qs + sw<D>(g8 + 8, 2 * ks + (t4 >> 1)) + off);
      qf[ks][0] = r0.x;
      qf[ks][1] = r1.x;
      qf[ks][2] = r0.y;
      qf[ks][3] = r1.y;
    }
  } else {
#pragma unroll
    for (int ks = 0; ks < KS; ++ks)
      ldmatrix_x4(qf[ks], smem_addr(qs) + sw<D>((lane & 7) + ((lane >> 3) & 1) * 8, 2 * ks + (lane >> 4)));
  }

  float o[ND][4];
#pragma unroll
  for (int nd = 0; nd < ND; ++nd)
#pragma unroll
    for (int k = 0; k < 4; ++k) o[nd][k] = 0.f;
  float m[2] = {kFloor, kFloor}, l[2] = {0.f, 0.f};
  // int8: the running maximum of the value weights' exponents (score + log2
  // of the value row's scale), less m, so the f16 weights never overflow
  float dmo[2] = {kFloor, kFloor};
  // int8: the accumulators' bias 1152 sum_k P of rows g, g + 8 (ob[0], ob[2])
  // and the scores' starting value -1152 sum_d Q (same rows), formed by the
  // MMA itself from the f16 query fragments
  float ob[4] = {0.f, 0.f, 0.f, 0.f};
  float kbias[2] = {0.f, 0.f};
  if constexpr (INT8) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) mma16<true>(acc, qf[ks], kF16x2_1152, kF16x2_1152);
    kbias[0] = -acc[0];
    kbias[1] = -acc[2];
  }
  // this lane's rows g and g + 8: tokens g / 4 and 2 + g / 4
  const int qpos[2] = {ctx + (lane >> 4), ctx + 2 + (lane >> 4)};

  bool aborted = false;
  int consumed = 0;
  for (int it = 0, kt = kt_begin; kt < kt_end; ++it, ++kt) {
    if (kt + C::kStages - 1 < kt_end) {
      load_part(kt + C::kStages - 1, (it + C::kStages - 1) % C::kStages);
      ++issued;
    }
    const int st = it % C::kStages;
    // (bounded: a copy that never lands leaves a status bit, not a hang)
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(&bars[st], (uint32_t)((it / C::kStages) & 1)))) {
      aborted = true;
      if (lane == 0) report(p, KVATTN_DEV_TIMEOUT);
      break;
    }
    consumed = it + 1;
    // a stage on an out-of-range page was not copied: nothing of it is used
    if ((bad >> st) & 1u) continue;
    const uint32_t kb = smem_addr(ring + st * C::kStage), vb = kb + C::kTile;
    const int key0 = kt * kPsKeys + wk;
    if constexpr (!INT8) {
      // bf16 rows past the keys hold whatever the pool holds (NaN, maybe):
      // zero them in V, so that their zero weights meet zeros
      const int nv = n_keys - key0;
      if (nv < kPsWarpKeys) {
        uint8_t *Vt = ring + st * C::kStage + C::kTile;
        const int n16 = (kPsWarpKeys - nv) * C::kRegions * 8;
        for (int idx = lane; idx < n16; idx += 32) {
          const int rr = nv + idx / (C::kRegions * 8), c = idx % (C::kRegions * 8);
          *reinterpret_cast<uint4 *>(Vt + (c >> 3) * C::kBox + rr * 128 + (c & 7) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        __syncwarp();
      }
    }
    if constexpr (INT8) {
      // Scores from the codes, which enter the MMAs as the f16 1152 + x (one
      // prmt a pair, the subtraction left to the accumulators): S = (Q codes^T)
      // * the key row's scale, starting from kbias = -1152 sum_d Q; value
      // weights 2^(S - m + log2 vs - dmo) with their own running maximum
      // m + dmo, so that P vs fits f16 whatever the scales and log2 vs is added
      // to a number near zero (the decode kernel's scheme); O accumulates
      // P (1152 + codes), whose bias 1152 sum_k P, formed by one more MMA with
      // a constant operand, ob takes, to be taken off at the end.  Lazy
      // references: m and dmo move only when a tile passes them by more than
      // kLazy, so the weights stay below 2^kLazy and most tiles leave the
      // accumulators as they are.
      const uint32_t kc = kb, vc = vb;
      const float *scl = wscl + st * 2 * kPsWarpKeys;
      // two accumulator chains per n-tile (k-steps c and c + 1), added at the
      // end: half the dependent MMAs in a row
      float s[2][4], s2[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          s[nt][e] = kbias[e >> 1];
          s2[nt][e] = 0.f;
        }
#pragma unroll
      for (int c = 0; c < D / 16; c += 2) {
        // matrices (keys 0-7, chunk c), (keys 0-7, c + 1), (keys 8-15, c),
        // (keys 8-15, c + 1); lane (g, t) holds codes 4t .. 4t + 3 of its key's
        // chunk: k-step c takes bytes 0, 1 as b0 and 2, 3 as b1
        const int kr = (lane & 7) + ((lane >> 4) << 3), ch = c + ((lane >> 3) & 1);
        uint32_t r[4];
        ldmatrix_x4(r, kc + (uint32_t)(kr * D + cidx8<D>(kr, ch) * 16));
        const uint32_t u00 = r[0] ^ 0x80808080u, u10 = r[2] ^ 0x80808080u;
        const uint32_t u01 = r[1] ^ 0x80808080u, u11 = r[3] ^ 0x80808080u;
        mma16<true>(s[0], qf[c], codes_biased_f16x2(u00, 0x5140u), codes_biased_f16x2(u00, 0x5342u));
        mma16<true>(s[1], qf[c], codes_biased_f16x2(u10, 0x5140u), codes_biased_f16x2(u10, 0x5342u));
        mma16<true>(s2[0], qf[c + 1], codes_biased_f16x2(u01, 0x5140u), codes_biased_f16x2(u01, 0x5342u));
        mma16<true>(s2[1], qf[c + 1], codes_biased_f16x2(u11, 0x5140u), codes_biased_f16x2(u11, 0x5342u));
      }
      // Lane (g, t) holds rows g, g + 8 (e / 2) at keys kr = 8 nt + 2t, + 1
      // (e % 2): each pair of a row shares its keys' scales (one 8-byte load
      // each), so the pair arithmetic is packed; a stage whose keys are all
      // cached ones (every row sees them) skips the causal mask.
      const bool whole = key0 + kPsWarpKeys - 1 <= ctx;
      float xv[2][4];  // log2 vs, then the value-weight exponents
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int kr = nt * 8 + 2 * (lane & 3);
        const float2 ks = *reinterpret_cast<const float2 *>(scl + kr);
        const float2 vs = *reinterpret_cast<const float2 *>(scl + kPsWarpKeys + kr);
        const float lv0 = lg2_approx(vs.x), lv1 = lg2_approx(vs.y);
        // (the two accumulator chains added first)
        const float2 a01 =
            mul_f32x2(add_f32x2(make_float2(s[nt][0], s[nt][1]), make_float2(s2[nt][0], s2[nt][1])), ks);
        const float2 a23 =
            mul_f32x2(add_f32x2(make_float2(s[nt][2], s[nt][3]), make_float2(s2[nt][2], s2[nt][3])), ks);
        s[nt][0] = a01.x;
        s[nt][1] = a01.y;
        s[nt][2] = a23.x;
        s[nt][3] = a23.y;
        xv[nt][0] = lv0;
        xv[nt][1] = lv1;
        xv[nt][2] = lv0;
        xv[nt][3] = lv1;
        if (!whole) {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (key0 + kr + (e & 1) > qpos[e >> 1]) {  // (keys past n_keys: past qpos)
              s[nt][e] = -INFINITY;
              xv[nt][e] = -INFINITY;
            }
        }
      }
      float mx[2] = {fmaxf(max3f(s[0][0], s[0][1], s[1][0]), s[1][1]),
                     fmaxf(max3f(s[0][2], s[0][3], s[1][2]), s[1][3])};
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xffffffffu, mx[rr], 1));
        mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xffffffffu, mx[rr], 2));
        if (mx[rr] > m[rr] + kLazy) {
          l[rr] *= ex2_approx(m[rr] - mx[rr]);
          dmo[rr] -= mx[rr] - m[rr];  // the same absolute reference
          m[rr] = mx[rr];
        }
      }
      // d = S - m, pair by pair; the value-weight exponents log2 vs + d
      float2 dd[2][2];  // [nt][row]
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        dd[nt][0] = sub_f32x2(s[nt][0], s[nt][1], m[0]);
        dd[nt][1] = sub_f32x2(s[nt][2], s[nt][3], m[1]);
        const float2 x01 = add_f32x2(make_float2(xv[nt][0], xv[nt][1]), dd[nt][0]);
        const float2 x23 = add_f32x2(make_float2(xv[nt][2], xv[nt][3]), dd[nt][1]);
        xv[nt][0] = x01.x;
        xv[nt][1] = x01.y;
        xv[nt][2] = x23.x;
        xv[nt][3] = x23.y;
      }
      float mxo[2] = {fmaxf(max3f(xv[0][0], xv[0][1], xv[1][0]), xv[1][1]),
                      fmaxf(max3f(xv[0][2], xv[0][3], xv[1][2]), xv[1][3])};
      float alpha_o[2] = {1.f, 1.f};
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        mxo[rr] = fmaxf(mxo[rr], __shfl_xor_sync(0xffffffffu, mxo[rr], 1));
        mxo[rr] = fmaxf(mxo[rr], __shfl_xor_sync(0xffffffffu, mxo[rr], 2));
        if (mxo[rr] > dmo[rr] + kLazy) {
          alpha_o[rr] = ex2_approx(dmo[rr] - mxo[rr]);
          dmo[rr] = mxo[rr];
        }
      }
      // the normaliser and the value weights from fp32 exponentials (an f16
      // pair exponential measured no faster); the weights, at most 2^kLazy, as
      // f16 pairs: the MMA's A fragment, rows g, g + 8 x keys 2t, 2t + 1 of
      // each n-tile (q: n-tile q / 2, row q % 2)
#pragma unroll
      for (int rr = 0; rr < 2; ++rr)
        l[rr] += (ex2_approx(dd[0][rr].x) + ex2_approx(dd[0][rr].y)) +
                 (ex2_approx(dd[1][rr].x) + ex2_approx(dd[1][rr].y));
      uint32_t a[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 w = sub_f32x2(xv[q >> 1][2 * (q & 1)], xv[q >> 1][2 * (q & 1) + 1], dmo[q & 1]);
        a[q] = pack16<true>(ex2_approx(w.x), ex2_approx(w.y));
      }
      if (__any_sync(0xffffffffu, alpha_o[0] != 1.f || alpha_o[1] != 1.f)) {
#pragma unroll
        for (int nd = 0; nd < ND; ++nd)
#pragma unroll
          for (int k = 0; k < 4; ++k) o[nd][k] *= alpha_o[k >> 1];
#pragma unroll
        for (int k = 0; k < 4; ++k) ob[k] *= alpha_o[k >> 1];
      }
      mma16<true>(ob, a, kF16x2_1152, kF16x2_1152);
#pragma unroll
      for (int c = 0; c < D / 16; c += 2) {
        // matrices (keys 0-7, chunk c), (keys 8-15, c), (keys 0-7, c + 1),
        // (keys 8-15, c + 1), transposed: lane (g, t) holds keys 2t, 2t + 1 at
        // dimensions 2g, 2g + 1 of the chunk; n-tile 2 c' takes the even
        // dimension (bytes 0, 2), 2 c' + 1 the odd one (bytes 1, 3)
        const int vr = (lane & 7) + ((lane >> 3) & 1) * 8, ch = c + (lane >> 4);
        uint32_t r[4];
        ldmatrix_x4_trans(r, vc + (uint32_t)(vr * D + cidx8<D>(vr, ch) * 16));
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int cc = c + h2;
          const uint32_t u0 = r[2 * h2] ^ 0x80808080u, u1 = r[2 * h2 + 1] ^ 0x80808080u;
          mma16<true>(o[2 * cc], a, codes_biased_f16x2(u0, 0x5240u), codes_biased_f16x2(u1, 0x5240u));
          mma16<true>(o[2 * cc + 1], a, codes_biased_f16x2(u0, 0x5341u), codes_biased_f16x2(u1, 0x5341u));
        }
      }
    } else {
      float s[2][4] = {};
  #pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        uint32_t kf[4];
        const int mi = lane >> 3;
        ldmatrix_x4(kf, kb + tile_sw<D>((mi >> 1) * 8 + (lane & 7), 2 * ks + (mi & 1)));
        mma16<INT8>(s[0], qf[ks], kf[0], kf[1]);
        mma16<INT8>(s[1], qf[ks], kf[2], kf[3]);
      }
      // the causal mask, skipped on a stage whose keys are all cached ones
      if (key0 + kPsWarpKeys - 1 > ctx) {
  #pragma unroll
        for (int nt = 0; nt < 2; ++nt)
  #pragma unroll
          for (int e = 0; e < 4; ++e)
            if (key0 + nt * 8 + 2 * (lane & 3) + (e & 1) > qpos[e >> 1])  // (keys past n_keys: past qpos)
              s[nt][e] = -INFINITY;
      }
      float mx[2] = {fmaxf(max3f(s[0][0], s[0][1], s[1][0]), s[1][1]),
                     fmaxf(max3f(s[0][2], s[0][3], s[1][2]), s[1][3])};
      // lazy reference: m moves only when a tile passes it by more than kLazy
      float alpha[2] = {1.f, 1.f};
  #pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xffffffffu, mx[rr], 1));
        mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xffffffffu, mx[rr], 2));
        if (mx[rr] > m[rr] + kLazy) {
          alpha[rr] = ex2_approx(m[rr] - mx[rr]);
          m[rr] = mx[rr];
          l[rr] *= alpha[rr];
        }
      }
      // weights 2^(S - m), the differences a row's pair at a time
      uint32_t a[4];
  #pragma unroll
      for (int q = 0; q < 4; ++q) {  // n-tile q / 2, row q % 2
        const float2 d = sub_f32x2(s[q >> 1][2 * (q & 1)], s[q >> 1][2 * (q & 1) + 1], m[q & 1]);
        const float w0 = ex2_approx(d.x), w1 = ex2_approx(d.y);
        l[q & 1] += w0 + w1;
        a[q] = pack16<INT8>(w0, w1);
      }
      if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
  #pragma unroll
        for (int nd = 0; nd < ND; ++nd)
  #pragma unroll
          for (int k = 0; k < 4; ++k) o[nd][k] *= alpha[k >> 1];
      }
  #pragma unroll
      for (int nd = 0; nd < ND; nd += 2) {
        uint32_t vf[4];
        ldmatrix_x4_trans(vf, vb + tile_sw<D>((lane & 7) + ((lane >> 3) & 1) * 8, nd + (lane >> 4)));
        mma16<INT8>(o[nd], a, vf[0], vf[1]);
        mma16<INT8>(o[nd + 1], a, vf[2], vf[3]);
      }
    }
    __syncwarp();  // the stage is rewritten C::kStages stages on
  }
  if (aborted && lane == 0) {
    // copies issued to slots no wait has looked at since are still in
    // flight: let them land before the warp leaves
    for (int i = consumed; i < issued; ++i)
      (void)mbar_wait_bounded(&bars[i % C::kStages], (uint32_t)((i / C::kStages) & 1));
  }
  cp_async_wait_all();
  if (!appended) pdl_wait_primary();
  pdl_launch_dependents();  // the merge grid may be placed
  __syncthreads();

  // ---- the four warps' states of each row: M = max m_w, weights 2^(m_w - M) ----
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    l[rr] += __shfl_xor_sync(0xffffffffu, l[rr], 1);
    l[rr] += __shfl_xor_sync(0xffffffffu, l[rr], 2);
  }
  float *obuf = reinterpret_cast<float *>(rings);  // [warp][row][D]
  float2 *ml = reinterpret_cast<float2 *>(obuf + kPfWarps * 16 * D);  // [warp][row]
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    const int r = (lane >> 2) + 8 * rr;
    if constexpr (INT8) {
      // o, less its bias, is relative to 2^(m + dmo): bring it to 2^m; n-tiles
      // 2 c and 2 c + 1 hold the even and odd dimensions of chunk c, this
      // lane's 16 c + 4t .. + 3
      const float f = ex2_approx(dmo[rr]), bias = ob[2 * rr];
      float *dst = obuf + (warp * 16 + r) * D + 4 * (lane & 3);
#pragma unroll
      for (int c = 0; c < D / 16; ++c)
        *reinterpret_cast<float4 *>(dst + 16 * c) =
            make_float4((o[2 * c][2 * rr] - bias) * f, (o[2 * c + 1][2 * rr] - bias) * f,
                        (o[2 * c][2 * rr + 1] - bias) * f, (o[2 * c + 1][2 * rr + 1] - bias) * f);
    } else {
      float *dst = obuf + (warp * 16 + r) * D + 2 * (lane & 3);
#pragma unroll
      for (int nd = 0; nd < ND; ++nd)
        *reinterpret_cast<float2 *>(dst + 8 * nd) = make_float2(o[nd][2 * rr], o[nd][2 * rr + 1]);
    }
    if ((lane & 3) == 0) ml[warp * 16 + r] = make_float2(m[rr], l[rr]);
  }
  __syncthreads();
  // one split: the output; several: this split's state, merged by
  // prefill_merge_kernel (a warp per row there hides the loads' latency better
  // than the last split to finish merging, or a CTA per head quad)
  const bool direct = p.n_splits == 1;
  // thread: row tid / 8 and columns cq + 32 k (cq = 4 (tid % 8)): the row's
  // weights once, then every load of its columns at once
  const int r = tid >> 3, cq = (tid & 7) * 4;
  const int t = r >> 2, h = h0 + (r & 3);
  if (t < n_new && t < kPsTok) {
    float2 st[kPfWarps];
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kPfWarps; ++w) {
      st[w] = ml[w * 16 + r];
      M = fmaxf(M, st[w].x);
    }
    float wt[kPfWarps], L = 0.f;
#pragma unroll
    for (int w = 0; w < kPfWarps; ++w) {
      wt[w] = ex2_approx(st[w].x - M);
      L += wt[w] * st[w].y;
    }
    float4 acc[D / 32];
#pragma unroll
    for (int k = 0; k < D / 32; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < kPfWarps; ++w)
#pragma unroll
      for (int k = 0; k < D / 32; ++k) {
        const float4 ov = *reinterpret_cast<const float4 *>(obuf + (w * 16 + r) * D + cq + 32 * k);
        acc[k].x += wt[w] * ov.x;
        acc[k].y += wt[w] * ov.y;
        acc[k].z += wt[w] * ov.z;
        acc[k].w += wt[w] * ov.w;
      }
    if (!direct) {
      // (records are D + 2 floats: 8-byte aligned)
      float *rec = p.part + (((size_t)z * p.n_tok + start + t) * p.n_qh + h) * (D + 2);
#pragma unroll
      for (int k = 0; k < D / 32; ++k) {
        *reinterpret_cast<float2 *>(rec + cq + 32 * k) = make_float2(acc[k].x, acc[k].y);
        *reinterpret_cast<float2 *>(rec + cq + 32 * k + 2) = make_float2(acc[k].z, acc[k].w);
      }
      if (cq == 0) *reinterpret_cast<float2 *>(rec + D) = make_float2(M, L);
    } else {
      const float f = L > 0.f ? 1.f / L : 0.f;
      __nv_bfloat16 *orow = p.out + ((size_t)(start + t) * p.n_qh + h) * D;
#pragma unroll
      for (int k = 0; k < D / 32; ++k)
        *reinterpret_cast<uint2 *>(orow + cq + 32 * k) =
            make_uint2(pack_bf16(acc[k].x * f, acc[k].y * f), pack_bf16(acc[k].z * f, acc[k].w * f));
    }
  }
}

// ---- merge of the splits' partial states -------------------------------------
// A warp per (new-token row, query head): M = max_z m_z, w_z = 2^(m_z - M),
// out = sum_z w_z o_z / sum_z w_z l_z (the blockwise softmax's recombination,
// "Qwen3-8B inference engine from scratch in C++/CUDA", section 4.4.1).
template <int D>
__global__ void __launch_bounds__(kPfThreads) prefill_merge_kernel(const __grid_constant__ PrefillParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_wait_primary();  // the attention grid's partial states are complete and visible
  const long long item = (long long)blockIdx.x * kPfWarps + warp;  // (row, query head)
  if (item >= (long long)p.n_tok * p.n_qh) return;
  const int r = (int)(item / p.n_qh), h = (int)(item - (long long)r * p.n_qh);
  const int lo = seq_of_row(p, r, lane);
  int start, n_new, ctx;
  // rows of skipped sequences, and past the tiles the grid covered, stay unwritten
  if (!seq_span(p, lo, start, n_new, ctx) || r < start || r >= start + n_new ||
      r - start >= p.tiles_per_seq * p.tile_rows)
    return;
  constexpr int E = D / 32;  // output columns per lane
  const size_t stride = (size_t)p.n_tok * p.n_qh * (D + 2);
  const float *rec = p.part + ((size_t)r * p.n_qh + h) * (D + 2);
  // the splits of the row's query tile, as the attention kernel formed them
  const int t0 = ((r - start) / p.tile_rows) * p.tile_rows;
  int nz;
  if (p.tile_rows == kPsTok) {
    nz = short_splits((short_tile_keys(ctx, n_new) + kPsKeys - 1) / kPsKeys, p.n_splits);
  } else if (p.tc_tiles) {
    const int n_rows = min(n_new, p.tiles_per_seq * p.tile_rows);
    const int tc0 = ((r - start) / kTcTok) * kTcTok;
    nz = tc_splits((tc_tile_keys(ctx, n_rows, tc0) + kTcKeys - 1) / kTcKeys, p.n_splits);
  } else {
    nz = tile_splits((query_tile_keys(ctx, n_new, t0) + kPfKeys - 1) / kPfKeys, p.n_splits);
  }
  float M = -INFINITY;
  for (int zz = 0; zz < nz; ++zz) M = fmaxf(M, __ldg(rec + zz * stride + D));
  float L = 0.f, acc[E] = {};
  for (int zz = 0; zz < nz; ++zz) {
    const float *rz = rec + zz * stride;
    const float w = ex2_approx(__ldg(rz + D) - M);
    L += w * __ldg(rz + D + 1);
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] += w * __ldg(rz + lane + 32 * e);
  }
  const float f = L > 0.f ? 1.f / L : 0.f;
  __nv_bfloat16 *dst = p.out + ((size_t)r * p.n_qh + h) * D;
#pragma unroll
  for (int e = 0; e < E; ++e) dst[lane + 32 * e] = __float2bfloat16_rn(acc[e] * f);
}

// a launch that may overlap the end of the stream's previous kernel (its
// threads wait for that kernel with griddepcontrol.wait)
template <class K, class P>
cudaError_t launch_pdl(K kern, dim3 grid, int smem, cudaStream_t stream, const P &p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kPfThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int D, bool INT8>
cudaError_t launch_prefill_t(const PrefillParams &p, cudaStream_t stream) {
  using C = PfCfg<D, INT8>;
  // (set on every call: the attribute belongs to the current device)
  cudaError_t err = cudaFuncSetAttribute(prefill_attn_kernel<D, INT8>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (err != cudaSuccess) return err;
  const long long items = (long long)p.n_tok * p.n_kvh;
  prefill_append_kernel<D, INT8><<<(unsigned)((items + kPfWarps - 1) / kPfWarps), kPfThreads, 0, stream>>>(p);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const dim3 grid((unsigned)((long long)p.n_seq * p.tiles_per_seq * (p.n_qh / kPfWarps)), 1u,
                  (unsigned)p.n_splits);
  if (p.tile_rows == kPsTok) {
    using S = PsCfg<D, INT8>;
    err = cudaFuncSetAttribute(prefill_short_kernel<D, INT8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               S::kSmem);
    if (err != cudaSuccess) return err;
    PsParams sp;
    sp.p = p;
    const long long rows = (long long)p.num_pages * p.n_kvh * p.page_size;
    if (!pool_tensor_map(&sp.tmap_k, p.k_pages, rows, D, INT8) ||
        !pool_tensor_map(&sp.tmap_v, p.v_pages, rows, D, INT8))
      return cudaErrorInvalidValue;  // the tensor map could not be encoded
    err = launch_pdl(prefill_short_kernel<D, INT8>, grid, S::kSmem, stream, sp);
    if (err != cudaSuccess) return err;
  } else if (p.tc_tiles) {
    // long prompts over a bf16 cache: the tcgen05 kernel (prefill_tc.cu)
    err = launch_prefill_tc(p, D, p.tiles_per_seq * kPfRows, stream);
    if (err != cudaSuccess) return err;
  } else {
    err = launch_pdl(prefill_attn_kernel<D, INT8>, grid, C::kSmem, stream, p);
    if (err != cudaSuccess) return err;
  }
  err = cudaGetLastError();
  if (err != cudaSuccess || p.n_splits == 1) return err;
  const long long rows = (long long)p.n_tok * p.n_qh;
  return launch_pdl(prefill_merge_kernel<D>, dim3((unsigned)((rows + kPfWarps - 1) / kPfWarps)), 0,
                    stream, p);
}

bool pf_aligned(const void *ptr, size_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

}  // namespace

// host frequency tables (kvattn_api.cu)
void rope_tables(float rope_theta, int head_dim, double *inv_freq, float2 *turns);

}  // namespace kvattn

namespace {
constexpr int kPfMaxSplits = 16;
size_t split_bytes(long long n_tok, int n_qh, int head_dim) {
  return (size_t)n_tok * n_qh * (head_dim + 2) * sizeof(float);
}
}  // namespace

extern "C" size_t kvattn_prefill_workspace_size(int n_tok, int n_qh, int head_dim) {
  if (n_tok < 0 || n_qh < 1 || (head_dim != 64 && head_dim != 128)) return 0;
  return kPfMaxSplits * split_bytes(n_tok, n_qh, head_dim);
}

extern "C" int kvattn_prefill(const void *q, const void *k_new, const void *v_new, void *k_pages,
                              void *v_pages, const int32_t *block_table,
                              const int32_t *seq_starts, const int32_t *ctx_lens, void *out,
                              int n_seq, int n_tok, int n_qh, int n_kvh, int head_dim,
                              int page_size, float rope_theta, float scale, int kv_dtype,
                              void *stream, int max_pages_per_seq, int num_pages,
                              float *k_scales, float *v_scales, int max_new_tokens,
                              uint32_t *dev_status, void *workspace, size_t workspace_bytes) {
  using namespace kvattn;
  if (kv_dtype != KVATTN_KV_BF16 && kv_dtype != KVATTN_KV_INT8) return KVATTN_EUNSUPPORTED;
  const bool int8 = kv_dtype == KVATTN_KV_INT8;
  if (n_seq < 0 || n_tok < 0 || n_qh < 1 || n_kvh < 1 || n_qh % n_kvh != 0 ||
      max_pages_per_seq < 1 || num_pages < 1 || max_new_tokens < 0)
    return KVATTN_EINVAL;
  if (!std::isfinite(scale) || std::isnan(rope_theta) || std::isinf(rope_theta))
    return KVATTN_EINVAL;
  if (head_dim != 64 && head_dim != 128) return KVATTN_EUNSUPPORTED;
  if ((n_qh / n_kvh) % kPfWarps != 0) return KVATTN_EUNSUPPORTED;  // 4 heads to a CTA
  if (page_size != 16 && page_size != 32 && page_size != 64 && page_size != 128 &&
      page_size != 256)
    return KVATTN_EUNSUPPORTED;
  if (n_seq > KVATTN_MAX_SEQS || n_qh > 1024) return KVATTN_EUNSUPPORTED;
  if ((long long)max_pages_per_seq * page_size > (long long)INT_MAX) return KVATTN_EUNSUPPORTED;
  if ((long long)num_pages * n_kvh * page_size > (long long)INT_MAX) return KVATTN_EUNSUPPORTED;
  const long long tiles = ((long long)max_new_tokens + kPfRows - 1) / kPfRows;
  // grid sizes: query tiles x head groups, and a warp per (new token, head)
  if ((long long)n_seq * tiles * (n_qh / kPfWarps) > (long long)INT_MAX ||
      (long long)n_tok * n_qh > (long long)kPfWarps * INT_MAX)
    return KVATTN_EUNSUPPORTED;
  if (n_seq == 0 || n_tok == 0 || max_new_tokens == 0) return KVATTN_OK;  // nothing to do
  if (!q || !k_new || !v_new || !k_pages || !v_pages || !block_table || !seq_starts ||
      !ctx_lens || !out)
    return KVATTN_EINVAL;
  if (!pf_aligned(q, 16) || !pf_aligned(k_new, 16) || !pf_aligned(v_new, 16) ||
      !pf_aligned(k_pages, 16) || !pf_aligned(v_pages, 16) || !pf_aligned(out, 4) ||
      !pf_aligned(block_table, 4) || !pf_aligned(seq_starts, 4) || !pf_aligned(ctx_lens, 4) ||
      (dev_status && !pf_aligned(dev_status, 4)) || (workspace && !pf_aligned(workspace, 16)))
    return KVATTN_EINVAL;
  if (int8 && (!k_scales || !v_scales || !pf_aligned(k_scales, 16) || !pf_aligned(v_scales, 16)))
    return KVATTN_EINVAL;
  PrefillParams p = {};
  p.q = static_cast<const __nv_bfloat16 *>(q);
  p.k_new = static_cast<const __nv_bfloat16 *>(k_new);
  p.v_new = static_cast<const __nv_bfloat16 *>(v_new);
  p.k_pages = k_pages;
  p.v_pages = v_pages;
  p.k_scales = int8 ? k_scales : nullptr;
  p.v_scales = int8 ? v_scales : nullptr;
  p.out = static_cast<__nv_bfloat16 *>(out);
  p.block_table = block_table;
  p.seq_starts = seq_starts;
  p.ctx_lens = ctx_lens;
  p.status = dev_status;
  p.n_seq = n_seq;
  p.n_tok = n_tok;
  p.n_qh = n_qh;
  p.n_kvh = n_kvh;
  p.page_size = page_size;
  for (int s = page_size; s > 1; s >>= 1) ++p.page_shift;
  p.max_pages = max_pages_per_seq;
  p.num_pages = num_pages;
  // short chunks (at most kPsTok new tokens a sequence) take the kernel whose
  // MMA rows are tokens x heads; the rest 16-token tiles
  const bool short_chunks = max_new_tokens <= kPsTok;
  p.tiles_per_seq = short_chunks ? 1 : (int)tiles;
  p.tile_rows = short_chunks ? kPsTok : kPfRows;
  // Splits of a query tile's key tiles: short chunks over long contexts
  // (speculative verification, small decode-like chunks) share them among up
  // to 16 CTAs (at least kPfMinTiles key tiles each; chunks of at most kPsTok
  // tokens kPsMinTiles stages on average, in splits that shrink from one to
  // the next), so every context streams at once;
  // long prompts, whose query tiles already fill the GPU, take one, as does a
  // call without a workspace.
  // Long prompts over a bf16 cache take the tcgen05 kernel (64-token query
  // tiles, one CTA an SM): their splits aim at two CTAs an SM.
  p.tc_tiles = (!int8 && !short_chunks && max_new_tokens > 64 && pf_aligned(out, 16)) ? 1 : 0;
  {
    int S = 1;
    if (max_new_tokens <= 64) {
      S = kPfMaxSplits;
    } else {
      int dev = 0, sms = 152;
      if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      const long long base =
          p.tc_tiles ? (long long)n_seq * ((tiles * kPfRows + kTcTok - 1) / kTcTok) * (n_qh / kPfWarps)
                     : (long long)n_seq * tiles * (n_qh / kPfWarps);
      const long long want = p.tc_tiles ? 2LL * sms : 4LL * sms;
      S = (int)std::min<long long>(kPfMaxSplits, std::max<long long>(1, (want + base - 1) / base));
    }
    const size_t per = split_bytes(n_tok, n_qh, head_dim);
    if (S > 1) S = workspace ? (int)std::min<size_t>((size_t)S, workspace_bytes / per) : 1;
    p.n_splits = std::max(1, S);
    p.part = static_cast<float *>(workspace);
  }
  p.use_rope = rope_theta > 0.0f ? 1 : 0;
  p.qscale = (float)((double)scale * 1.4426950408889634);
  rope_tables(rope_theta, head_dim, p.inv_freq, p.turns);
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const cudaError_t err = head_dim == 64 ? (int8 ? launch_prefill_t<64, true>(p, st) : launch_prefill_t<64, false>(p, st))
                                         : (int8 ? launch_prefill_t<128, true>(p, st) : launch_prefill_t<128, false>(p, st));
  return err == cudaSuccess ? KVATTN_OK : cuda_fail(err);
}
