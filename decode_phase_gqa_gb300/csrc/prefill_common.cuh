// Pieces the prefill kernels share (prefill.cu: append, the mma.sync
// attention kernels and the merge; prefill_tc.cu: the tcgen05 attention
// kernel): launch constants, the kernel parameter block and the per-sequence
// span check.
#pragma once

#include "decode_common.cuh"

namespace kvattn {

constexpr int kPfWarps = 4;                  // query heads per CTA, one warp each
constexpr int kPfThreads = 32 * kPfWarps;
constexpr int kPfRows = 16;                  // new tokens per CTA (the MMA's M)
constexpr int kPfKeys = 32;                  // keys per staged tile
constexpr int kPfNT = kPfKeys / 8;           // its n-tiles of 8 keys (Q K^T)
constexpr int kPfKK = kPfKeys / 16;          // its k-steps of 16 keys (P V)
constexpr int kPfMinTiles = 16;              // key tiles a split takes at least
// short chunks (at most 4 new tokens a sequence: speculative drafts)
constexpr int kPsTok = 4;                    // new tokens a CTA (x 4 heads: the MMA's 16 rows)
constexpr int kPsWarpKeys = 16;              // keys of a stage each warp takes
constexpr int kPsKeys = kPfWarps * kPsWarpKeys;  // keys a stage holds
constexpr int kPsStages = 2;
constexpr int kPsMinTiles = 20;              // stages a split takes, on average, at least

// the tcgen05 attention kernel (prefill_tc.cu): 64 new tokens x 4 heads (two
// halves of 128 MMA rows) a CTA, 128-key tiles, splits of at least 4 tiles
constexpr int kTcTok = 64;
constexpr int kTcKeys = 128;
constexpr int kTcMinTiles = 4;

struct PrefillParams {
  const __nv_bfloat16 *q, *k_new, *v_new;
  void *k_pages, *v_pages;  // bf16, or int8 codes with k_scales / v_scales
  float *k_scales, *v_scales;
  __nv_bfloat16 *out;
  const int32_t *block_table, *seq_starts, *ctx_lens;
  uint32_t *status;  // KVATTN_DEV_* bits (NULL: not reported)
  int n_seq, n_tok, n_qh, n_kvh, page_size, page_shift, max_pages, num_pages;
  int tiles_per_seq;  // query tiles the grid gives each sequence
  int tile_rows;      // new tokens a query tile holds: 16, or kPsTok (short chunks)
  int n_splits;       // CTAs sharing one query tile's key tiles
  float *part;        // n_splits > 1: [n_splits][n_tok][n_qh][D + 2] partial
                      // states (o relative to 2^m, m, l; log2 units)
  int tc_tiles;       // the attention kernel is the tcgen05 one (64-token query
                      // tiles of 128-key tiles; the merge recomputes its splits);
                      // the append kernel then writes the rotated, scaled bf16
                      // query rows into out, where that kernel reads them
  int use_rope;
  float qscale;       // scale * log2(e)
  float2 turns[64];   // rope_theta^(-2i/d) / (2 pi) as fp32 head + remainder
  double inv_freq[64];
};

// ---- packed fp32 arithmetic (one instruction for a pair) ----------------------
// max(a, b, c) in one instruction
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
// (x0 - m, x1 - m), a + b and a * b by packed fp32 instructions, rounded as
// the scalar ones
__device__ __forceinline__ float2 sub_f32x2(float x0, float x1, float m) {
  float2 o;
  asm("{\n\t.reg .b64 x, y, r;\n\tmov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %4};\n\t"
      "sub.rn.f32x2 r, x, y;\n\tmov.b64 {%0, %1}, r;\n\t}"
      : "=f"(o.x), "=f"(o.y)
      : "f"(x0), "f"(x1), "f"(m));
  return o;
}
__device__ __forceinline__ float2 add_f32x2(float2 a, float2 b) {
  float2 o;
  asm("{\n\t.reg .b64 x, y, r;\n\tmov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %5};\n\t"
      "add.rn.f32x2 r, x, y;\n\tmov.b64 {%0, %1}, r;\n\t}"
      : "=f"(o.x), "=f"(o.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return o;
}
__device__ __forceinline__ float2 mul_f32x2(float2 a, float2 b) {
  float2 o;
  asm("{\n\t.reg .b64 x, y, r;\n\tmov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %5};\n\t"
      "mul.rn.f32x2 r, x, y;\n\tmov.b64 {%0, %1}, r;\n\t}"
      : "=f"(o.x), "=f"(o.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return o;
}
__device__ __forceinline__ void report(const PrefillParams &p, uint32_t bits) {
  if (p.status) atomicOr(p.status, bits);
}

// Sequence b's rows of the new-token arrays [start, start + n_new) and cached
// count ctx; false when they do not fit the arrays or the block table.
__device__ __forceinline__ bool seq_span(const PrefillParams &p, int b, int &start, int &n_new,
                                         int &ctx) {
  start = __ldg(p.seq_starts + b);
  const int end = __ldg(p.seq_starts + b + 1);
  ctx = __ldg(p.ctx_lens + b);
  n_new = end - start;
  const long long cap = (long long)p.max_pages << p.page_shift;
  return start >= 0 && end <= p.n_tok && n_new >= 0 && ctx >= 0 && (long long)ctx + n_new <= cap;
}

// The tcgen05 kernel's query tile starting at new token t0 (n_rows new tokens
// attended, after ctx cached ones): the keys its last row sees, and the
// splits sharing its 128-key tiles (at most S, each of at least kTcMinTiles).
__device__ __forceinline__ int tc_tile_keys(int ctx, int n_rows, int t0) {
  return ctx + min(n_rows, t0 + kTcTok);
}
__device__ __forceinline__ int tc_splits(int n_tiles, int S) {
  return max(1, min(S, (n_tiles + kTcMinTiles - 1) / kTcMinTiles));
}

// Launch of the tcgen05 attention kernel (prefill_tc.cu) for the long-prompt
// path over a bf16 cache: new tokens 0 .. cover - 1 of every sequence in
// 64-token query tiles, p.n_splits splits at most; the append kernel has been
// queued before it.
cudaError_t launch_prefill_tc(const PrefillParams &p, int head_dim, int cover,
                              cudaStream_t stream);

// The pools' TMA view used by the decode kernel (kvattn_api.cu): [rows][head_dim]
// with [16 rows][128 bytes] boxes, 128-byte swizzle (cached per pool).
bool pool_tensor_map(CUtensorMap *map, const void *base, long long rows, int head_dim, bool int8);

}  // namespace kvattn
