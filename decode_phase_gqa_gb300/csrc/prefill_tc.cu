// Long-prompt prefill attention on the fifth-generation tensor cores
// (tcgen05): the FlashAttention-2 blocking of "Qwen3-8B inference engine from
// scratch in C++/CUDA", section 4.4.1 (key blocks, a running maximum and
// normaliser per row, never the whole score matrix), with the causal mask of
// "LLM inference from smollm3.go", section "Prefill: the whole prompt at once"
// (new token i of a sequence attends over keys 0 .. ctx + i).
//
// A CTA owns 128 MMA rows: 32 new tokens of one sequence x the 4 query heads
// of one group (row 32 hh + tl: head hh of the group, token tl), so every
// staged K/V tile serves the whole group (section 4.4.2 of the Qwen3-8B page).
// Keys come in tiles of 64.  Six warps:
//   * warps 0-3 (one thread per row, TMEM lanes 32 w ..): rotate and scale the
//     query rows into shared memory; per tile read the scores S from tensor
//     memory, mask them, keep the row's running maximum m and normaliser l
//     (log2 units; the maximum moves lazily, by more than 8, so the
//     accumulator is rarely rescaled), write P = 2^(S - m) as bf16 into
//     shared memory; at the end read O, divide by l, store bf16;
//   * warp 4: TMA tensor copies of the K and V tiles (16-key page blocks,
//     [16 rows][128 bytes] boxes, 128-byte swizzle) into a 3-stage ring;
//   * warp 5, one thread: issues the MMAs, S = Q K^T into one of two TMEM
//     score buffers (M 128, N 64, K d) and O += P V into the TMEM accumulator
//     (M 128, N 64 per half of d, K 64), and commits them to mbarriers.
// S of tile i + 1 is computed while the softmax warps work on tile i; P is
// double-buffered so that the softmax of tile i + 1 need not wait for the
// P V products of tile i.  Every wait is bounded (KVATTN_DEV_TIMEOUT).
#include "prefill_common.cuh"

namespace kvattn {

namespace {

constexpr int kTcRows = 4 * kTcTok;  // MMA M: 32 new tokens x 4 heads
constexpr int kTcStages = 3;        // K/V tiles in flight
constexpr int kTcThreads = 192;
constexpr uint32_t kTmemCols = 256; // S[2][64] + O[d]

template <int D>
struct TcCfg {
  static constexpr int kRegions = D / 64;                    // 128-byte column blocks of a row
  static constexpr int kQRegion = kTcRows * 128;             // [128 rows][128 B]
  static constexpr int kKVRegion = kTcKeys * 128;            // [64 keys][128 B]
  static constexpr int kTile = kRegions * kKVRegion;         // K or V tile
  static constexpr int kStage = 2 * kTile;                   // K then V
  static constexpr int kPBuf = kTcRows * 128;                // P [128 rows][64 keys] bf16
  static constexpr int kQOff = 0;
  static constexpr int kStageOff = kQOff + kRegions * kQRegion;
  static constexpr int kPOff = kStageOff + kTcStages * kStage;
  static constexpr int kBarOff = kPOff + 2 * kPBuf;
  // full[S], empty[S], s_full[2], s_free[2], p_full[2], o_done[2], q_ready, mma_done
  static constexpr int kNumBars = 2 * kTcStages + 10;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;    // tmem base, abort flag, counters
  static constexpr int kTurnsOff = kMiscOff + 64;            // float2[64]
  static constexpr int kSmem = kTurnsOff + 512 + 1024;       // + slack for 1024-byte alignment
  static constexpr uint32_t kOCol = 128;                     // O's first TMEM column
  static_assert(kSmem <= 227 * 1024, "shared memory");
  static_assert(kStageOff % 1024 == 0 && kStage % 1024 == 0 && kPOff % 1024 == 0,
                "swizzle atoms need 1024-byte alignment");
};

struct PfTcParams {
  CUtensorMap tmap_k, tmap_v;  // [rows][D] bf16 pools, [16][64] boxes, 128-byte swizzle
  PrefillParams p;
  int n_qt;   // 32-token query tiles per sequence
  int cover;  // new tokens of a sequence the launch covers
};

// ---- tcgen05 / TMEM wrappers ---------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t *slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(slot)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D (TMEM, fp32) = A B (+ D when acc): A and B bf16 in shared memory
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(acc)
      : "memory");
}
// `bar` receives one arrival when every tcgen05 operation this thread issued
// before has completed
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_addr(bar))
               : "memory");
}

// Shared-memory matrix descriptor of a 128-byte-swizzled operand: start
// address, leading and stride byte offsets (16-byte units), the fixed 0b001 of
// bits 46-48, swizzle mode 2 (128 bytes) in bits 61-63.  The start may move by
// 32-byte steps inside a 1024-byte swizzle atom (the swizzle is a function of
// the address bits, so the K offset of an MMA is a plain add).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulator (bits 4-5 = 1), A and
// B bf16 (bits 7-9, 10-12 = 1), A K-major, B K-major or MN-major (bit 16),
// N / 8 in bits 17-22, M / 16 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Columns c .. c + 31 of this thread's TMEM lane (32x32b shape: thread i
// of the warp reads lane 32 (warp % 4) + i), as fp32; the wait for the load is
// in the same statement, so no use of r can be scheduled before it.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Columns c .. c + 63 of this thread's TMEM lane (32x32b shape: thread i
// of the warp reads lane 32 (warp % 4) + i), as fp32; the wait for the load is
// in the same statement, so no use of r can be scheduled before it.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
        "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
        "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

// Store columns c .. c + 31 of this thread's TMEM lane and wait for the
// stores to complete.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n\t"
      "tcgen05.wait::st.sync.aligned;"
      :
      : "r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
        "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])), "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])), "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
        "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}


// TMA tensor copy with the default L2 policy: the tiles of a sequence are read
// again by every later query tile of it
__device__ __forceinline__ void tma_load_2d_keep(void *dst, const CUtensorMap *map, int x, int y,
                                                 uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

// Bounded wait on an mbarrier phase by one thread; on a timeout the CTA's
// abort flag is set and KVATTN_DEV_TIMEOUT reported.
__device__ __forceinline__ bool tc_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                        const PrefillParams &p) {
  if (mbar_wait_bounded(bar, parity)) return true;
  *abort_flag = 1;
  report(p, KVATTN_DEV_TIMEOUT);
  return false;
}

template <int D>
__global__ void __launch_bounds__(kTcThreads, 1) prefill_tc_kernel(const __grid_constant__ PfTcParams tp) {
  using C = TcCfg<D>;
  const PrefillParams &p = tp.p;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // CTA x: head quad x % G, then sequence, then query tile from the last (the
  // tiles with the most keys start first)
  const int G = p.n_qh / kPfWarps;
  const int grp = (int)(blockIdx.x % G), rest = (int)(blockIdx.x / G);
  const int b = rest % p.n_seq, qt = tp.n_qt - 1 - rest / p.n_seq;
  const int g = p.n_qh / p.n_kvh;
  const int j = grp / (g / kPfWarps);
  const int h0 = j * g + (grp % (g / kPfWarps)) * kPfWarps;
  int start, n_new, ctx;
  // (every early exit below is the same for the whole CTA; each thread waits
  // for the append grid before it leaves)
  if (!seq_span(p, b, start, n_new, ctx)) {
    if (qt == 0 && grp == 0 && tid == 0) report(p, KVATTN_DEV_BAD_LEN);
    pdl_wait_primary();
    return;
  }
  if (qt == 0 && grp == 0 && tid == 0 && n_new > tp.cover) report(p, KVATTN_DEV_BAD_LEN);
  const int n_rows_tok = min(n_new, tp.cover);  // new tokens the launch attends
  const int t0 = qt * kTcTok;
  if (t0 >= n_rows_tok) {
    pdl_wait_primary();
    return;
  }
  const int n_keys = tc_tile_keys(ctx, n_rows_tok, t0);  // keys the tile's last row sees
  const int all_tiles = (n_keys + kTcKeys - 1) / kTcKeys;
  // split z of the query tile takes a contiguous range of its key tiles (a
  // split past the tile's count has nothing to do)
  const int z = (int)blockIdx.z, nz = tc_splits(all_tiles, p.n_splits);
  if (z >= nz) {
    pdl_wait_primary();
    return;
  }
  const int per = (all_tiles + nz - 1) / nz;
  const int kt0 = min(all_tiles, z * per);
  const int n_tiles = min(all_tiles, kt0 + per) - kt0;  // may be 0: an empty partial state

  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kBarOff);
  uint64_t *full = bars, *empty = bars + kTcStages;
  uint64_t *s_full = bars + 2 * kTcStages, *s_free = s_full + 2, *p_full = s_free + 2;
  uint64_t *o_done = p_full + 2, *q_ready = o_done + 2, *mma_done = q_ready + 1;
  uint32_t *misc = reinterpret_cast<uint32_t *>(smem + C::kMiscOff);
  uint32_t *tmem_slot = misc;                                 // [0]
  volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + 1);
  volatile int *issued_tiles = reinterpret_cast<volatile int *>(misc + 2);
  float2 *turns = reinterpret_cast<float2 *>(smem + C::kTurnsOff);
  uint8_t *qs = smem + C::kQOff;
  uint8_t *stages = smem + C::kStageOff;
  uint8_t *pbuf = smem + C::kPOff;

  if (tid == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], kTcRows);
      mbar_init(&p_full[i], kTcRows);
      mbar_init(&o_done[i], 1);
    }
    mbar_init(q_ready, kTcRows);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    *issued_tiles = 0;
    fence_barrier_init();
  }
  if (tid < 64) turns[tid] = p.turns[tid];
  if (warp == 0) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
    // ---- softmax warps: one thread per row ------------------------------------
    const int row = tid;  // 32 warp + lane: head h0 + warp, token t0 + lane
    const int h = h0 + warp, t = t0 + lane;
    const bool live = t < n_rows_tok;
    // the row's query, rotated in fp32 at position ctx + t, scaled by
    // scale * log2(e), rounded to bf16, into the swizzled Q tile
    {
      const uint4 *src = reinterpret_cast<const uint4 *>(p.q + ((size_t)(start + (live ? t : 0)) * p.n_qh + h) * D);
#pragma unroll 1
      for (int c = 0; c < D / 16; ++c) {
        uint4 lo4 = make_uint4(0u, 0u, 0u, 0u), hi4 = lo4;
        if (live) {
          lo4 = src[c];
          hi4 = src[c + D / 16];
        }
        const uint32_t lw[4] = {lo4.x, lo4.y, lo4.z, lo4.w}, hw[4] = {hi4.x, hi4.y, hi4.z, hi4.w};
        uint32_t ol[4], oh[4];
#pragma unroll
        for (int e2 = 0; e2 < 4; ++e2) {
          float a[2], bb[2];
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int i = 8 * c + 2 * e2 + k;
            float lo = __uint_as_float(k ? (lw[e2] & 0xffff0000u) : (lw[e2] << 16));
            float hi = __uint_as_float(k ? (hw[e2] & 0xffff0000u) : (hw[e2] << 16));
            if (p.use_rope && live) {
              float sn, cs;
              sincospif(2.f * frac_turns(ctx + t, turns[i]), &sn, &cs);
              const float x = lo * cs - hi * sn, y = hi * cs + lo * sn;
              lo = x;
              hi = y;
            }
            a[k] = lo * p.qscale;
            bb[k] = hi * p.qscale;
          }
          ol[e2] = pack_bf16(a[0], a[1]);
          oh[e2] = pack_bf16(bb[0], bb[1]);
        }
        const int il = 8 * c, ih = 8 * c + D / 2;  // first element of each chunk
        uint8_t *dl = qs + (il / 64) * C::kQRegion + row * 128 + ((((il % 64) / 8) ^ (row & 7)) << 4);
        uint8_t *dh = qs + (ih / 64) * C::kQRegion + row * 128 + ((((ih % 64) / 8) ^ (row & 7)) << 4);
        *reinterpret_cast<uint4 *>(dl) = make_uint4(ol[0], ol[1], ol[2], ol[3]);
        *reinterpret_cast<uint4 *>(dh) = make_uint4(oh[0], oh[1], oh[2], oh[3]);
      }
    }
    fence_proxy_async_smem();  // the MMAs read Q through the async proxy
    mbar_arrive(q_ready);
    pdl_wait_primary();

    const uint32_t lane_base = tmem + ((uint32_t)(32 * warp) << 16);
    const int kmax = live ? ctx + t : -1;  // last key the row sees
    const float kFloor = -1e30f;
    float m_run = kFloor, l_run = 0.f;
    int i = 0;
    for (; i < n_tiles; ++i) {
      if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
      const int buf = i & 1;
      if (!__all_sync(0xffffffffu, tc_wait(&s_full[buf], (uint32_t)((i >> 1) & 1), abort_flag, p))) break;
      tc_fence_after();
      float s[kTcKeys];
      tmem_ld64(lane_base + (uint32_t)(buf * kTcKeys), s);
      tc_fence_before();
      mbar_arrive(&s_free[buf]);
      // masks: causal (key <= ctx + t), and pages outside the pool
      const int key0 = (kt0 + i) * kTcKeys;
      bool gv[kTcKeys / 16];
#pragma unroll
      for (int q4 = 0; q4 < kTcKeys / 16; ++q4) {
        const int key = key0 + 16 * q4;
        bool ok = key <= kmax;
        if (ok) {
          const int pg = __ldg(p.block_table + (size_t)b * p.max_pages + (key >> p.page_shift));
          ok = pg >= 0 && pg < p.num_pages;
        }
        gv[q4] = ok;
      }
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < kTcKeys; ++c) {
        const bool ok = gv[c >> 4] && key0 + c <= kmax;
        s[c] = ok ? s[c] : -INFINITY;
        mx = fmaxf(mx, s[c]);
      }
      const float m_new = fmaxf(m_run, mx);
      const bool need = m_new > m_run + 8.f;
      const float alpha = need ? ex2_approx(m_run - m_new) : 1.f;
      if (i > 0 && __any_sync(0xffffffffu, need)) {
        // rescale this warp's rows of O once the P V products of tile i - 1 are in
        if (!__all_sync(0xffffffffu, tc_wait(&o_done[(i - 1) & 1], (uint32_t)(((i - 1) >> 1) & 1), abort_flag, p)))
          break;
        tc_fence_after();
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          float o[32];
          tmem_ld32(lane_base + C::kOCol + (uint32_t)c0, o);
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] *= alpha;
          tmem_st32(lane_base + C::kOCol + (uint32_t)c0, o);
        }
      }
      if (need) {
        m_run = m_new;
        l_run *= alpha;
      }
      // The last tile may end inside a 16-key block whose rows past the keys
      // hold whatever the pool has there (possibly not a number): zero those V
      // rows, so that their zero weights cannot meet a NaN in the MMA (the
      // masked scores are selected away, so stale K rows do no harm).
      if (kt0 + i == all_tiles - 1 && (n_keys & 15) != 0) {
        const int s = i % kTcStages;
        if (!__all_sync(0xffffffffu, tc_wait(&full[s], (uint32_t)((i / kTcStages) & 1), abort_flag, p)))
          break;
        const int r0 = n_keys - key0, r1 = (r0 + 15) & ~15;
        uint8_t *vt = stages + s * C::kStage + C::kTile;
        for (int e = tid; e < (r1 - r0) * C::kRegions * 8; e += kTcRows) {
          const int r = r0 + e / (C::kRegions * 8), rest = e % (C::kRegions * 8);
          *reinterpret_cast<uint4 *>(vt + (rest >> 3) * C::kKVRegion + r * 128 + (rest & 7) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
      }
      // P buffer buf is free once the P V products of tile i - 2 are in
      if (i >= 2 &&
          !__all_sync(0xffffffffu, tc_wait(&o_done[buf], (uint32_t)(((i >> 1) - 1) & 1), abort_flag, p)))
        break;
      uint8_t *prow = pbuf + buf * C::kPBuf + row * 128;
#pragma unroll
      for (int c8 = 0; c8 < kTcKeys / 8; ++c8) {
        uint32_t w[4];
#pragma unroll
        for (int e2 = 0; e2 < 4; ++e2) {
          const __nv_bfloat162 pr = __floats2bfloat162_rn(ex2_approx(s[8 * c8 + 2 * e2] - m_run),
                                                          ex2_approx(s[8 * c8 + 2 * e2 + 1] - m_run));
          const float2 pf = __bfloat1622float2(pr);
          l_run += pf.x + pf.y;  // the normaliser of the weights the MMA uses
          w[e2] = *reinterpret_cast<const uint32_t *>(&pr);
        }
        *reinterpret_cast<uint4 *>(prow + ((c8 ^ (row & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&p_full[buf]);
    }
    // ---- the row's output: O / l rounded to bf16, or (several splits) the
    // partial state o (relative to 2^m), m, l for the merge kernel ------------
    if (i == n_tiles) {
      const int last = n_tiles - 1;
      const bool ok = n_tiles == 0 ||
                      __all_sync(0xffffffffu, tc_wait(&o_done[last & 1], (uint32_t)((last >> 1) & 1), abort_flag, p));
      if (ok) {
        if (n_tiles > 0) tc_fence_after();
        const float f = l_run > 0.f ? 1.f / l_run : 0.f;  // no visible key: a zero row
        __nv_bfloat16 *dst = p.out + ((size_t)(start + (live ? t : 0)) * p.n_qh + h) * D;
        float *rec = p.part + (((size_t)z * p.n_tok + start + (live ? t : 0)) * p.n_qh + h) * (D + 2);
        const bool split = p.n_splits > 1;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          float o[32];
          if (n_tiles > 0) {
            tmem_ld32(lane_base + C::kOCol + (uint32_t)c0, o);
          } else {
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] = 0.f;
          }
          if (live && split) {
#pragma unroll
            for (int k = 0; k < 32; k += 2)
              *reinterpret_cast<float2 *>(rec + c0 + k) = make_float2(o[k], o[k + 1]);
          } else if (live) {
#pragma unroll
            for (int k = 0; k < 32; k += 8) {
              const uint4 v = make_uint4(pack_bf16(o[k] * f, o[k + 1] * f), pack_bf16(o[k + 2] * f, o[k + 3] * f),
                                         pack_bf16(o[k + 4] * f, o[k + 5] * f), pack_bf16(o[k + 6] * f, o[k + 7] * f));
              *reinterpret_cast<uint4 *>(dst + c0 + k) = v;
            }
          }
        }
        if (live && split) *reinterpret_cast<float2 *>(rec + D) = make_float2(m_run, l_run);
      }
    }
    tc_fence_before();
  } else if (warp == 4) {
    // ---- producer: K and V tiles by TMA ----------------------------------------------
    pdl_wait_primary();  // the appended rows are complete and visible
    prefetch_tensormap(&tp.tmap_k);
    prefetch_tensormap(&tp.tmap_v);
    int i = 0;
    for (; i < n_tiles; ++i) {
      if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
      const int s = i % kTcStages;
      if (i >= kTcStages) {
        bool ok = true;
        if (lane == 0) ok = tc_wait(&empty[s], (uint32_t)(((i / kTcStages) - 1) & 1), abort_flag, p);
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      }
      // pool row of each 16-key block of the tile (lanes 0-3); rows past the
      // keys or on an out-of-range page are fetched from row -16, outside the
      // view, which the copy fills with zeros
      int prow = -16;
      if (lane < kTcKeys / 16) {
        const int key = (kt0 + i) * kTcKeys + 16 * lane;
        if (key < n_keys) {
          const int pg = __ldg(p.block_table + (size_t)b * p.max_pages + (key >> p.page_shift));
          if (pg >= 0 && pg < p.num_pages)
            prow = (pg * p.n_kvh + j) * p.page_size + (key & (p.page_size - 1));
          else
            report(p, KVATTN_DEV_BAD_PAGE);
        }
      }
      int rows[kTcKeys / 16];
#pragma unroll
      for (int q4 = 0; q4 < kTcKeys / 16; ++q4) rows[q4] = __shfl_sync(0xffffffffu, prow, q4);
      if (lane == 0) {
        uint8_t *kd = stages + s * C::kStage, *vd = kd + C::kTile;
        mbar_arrive_expect_tx(&full[s], C::kStage);
#pragma unroll
        for (int q4 = 0; q4 < kTcKeys / 16; ++q4)
#pragma unroll
          for (int r = 0; r < C::kRegions; ++r) {
            tma_load_2d_keep(kd + r * C::kKVRegion + q4 * 2048, &tp.tmap_k, 64 * r, rows[q4], &full[s]);
            tma_load_2d_keep(vd + r * C::kKVRegion + q4 * 2048, &tp.tmap_v, 64 * r, rows[q4], &full[s]);
          }
        *issued_tiles = i + 1;
      }
      __syncwarp();
    }
  } else {
    // ---- MMA issuer: one thread -------------------------------------------------------
    pdl_wait_primary();
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16(kTcRows, kTcKeys, false);
      constexpr uint32_t kIdPV = idesc_bf16(kTcRows, 64, true);
      const uint32_t q0 = smem_addr(qs), st0 = smem_addr(stages), p0 = smem_addr(pbuf);
      bool ok = tc_wait(q_ready, 0, abort_flag, p);
      tc_fence_after();
      auto issue_s = [&](int i) -> bool {
        const int s = i % kTcStages, buf = i & 1;
        if (!tc_wait(&full[s], (uint32_t)((i / kTcStages) & 1), abort_flag, p)) return false;
        if (i >= 2 && !tc_wait(&s_free[buf], (uint32_t)(((i >> 1) - 1) & 1), abort_flag, p)) return false;
        tc_fence_after();
        const uint32_t kb = st0 + (uint32_t)(s * C::kStage);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (uint32_t)((ks & 3) * 32);  // 16 elements on, inside the atom
          const uint64_t a = sw128_desc(q0 + (uint32_t)((ks >> 2) * C::kQRegion) + off, 16, 1024);
          const uint64_t bd = sw128_desc(kb + (uint32_t)((ks >> 2) * C::kKVRegion) + off, 16, 1024);
          tc_mma(tmem + (uint32_t)(buf * kTcKeys), a, bd, kIdS, ks > 0 ? 1u : 0u);
        }
        tc_commit(&s_full[buf]);
        return true;
      };
      auto issue_pv = [&](int i) -> bool {
        const int s = i % kTcStages, buf = i & 1;
        if (!tc_wait(&p_full[buf], (uint32_t)((i >> 1) & 1), abort_flag, p)) return false;
        tc_fence_after();
        const uint32_t vb = st0 + (uint32_t)(s * C::kStage + C::kTile);
        const uint32_t pa = p0 + (uint32_t)(buf * C::kPBuf);
#pragma unroll
        for (int hf = 0; hf < C::kRegions; ++hf)
#pragma unroll
          for (int ks = 0; ks < kTcKeys / 16; ++ks) {
            const uint64_t a = sw128_desc(pa + (uint32_t)(ks * 32), 16, 1024);
            // V: [keys][64 d] per half, rows of d contiguous (MN-major for B);
            // 16 keys = two 8-row groups = 2048 bytes on
            const uint64_t bd = sw128_desc(vb + (uint32_t)(hf * C::kKVRegion + ks * 2048), 1024, 1024);
            tc_mma(tmem + C::kOCol + (uint32_t)(64 * hf), a, bd, kIdPV, (i > 0 || ks > 0) ? 1u : 0u);
          }
        tc_commit(&o_done[buf]);
        tc_commit(&empty[s]);
        return true;
      };
      if (ok && n_tiles > 0) ok = issue_s(0);
      if (ok && n_tiles > 1) ok = issue_s(1);
      for (int i = 0; ok && i < n_tiles; ++i) {
        if (*abort_flag) break;
        ok = issue_pv(i);
        if (ok && i + 2 < n_tiles) ok = issue_s(i + 2);
      }
      // every MMA issued has completed before the tensor memory is freed
      tc_commit(mma_done);
      (void)tc_wait(mma_done, 0, abort_flag, p);
    }
    __syncwarp();
  }

  __syncthreads();
  if (warp == 4 && lane == 0 && *abort_flag) {
    // copies still in flight on a stage nobody waited for land before the CTA leaves
    const int n = *issued_tiles;
    for (int i = max(0, n - kTcStages); i < n; ++i)
      (void)mbar_wait_bounded(&full[i % kTcStages], (uint32_t)((i / kTcStages) & 1));
  }
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

template <int D>
cudaError_t launch_tc_t(const PfTcParams &tp, cudaStream_t stream) {
  using C = TcCfg<D>;
  cudaError_t err = cudaFuncSetAttribute(prefill_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmem);
  if (err != cudaSuccess) return err;
  const long long ctas = (long long)tp.p.n_seq * tp.n_qt * (tp.p.n_qh / kPfWarps);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ctas, 1u, (unsigned)tp.p.n_splits);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = (size_t)C::kSmem;
  cfg.stream = stream;
  // a programmatic dependent of the append kernel: the queries are formed while
  // it runs; every thread waits for it before reading keys or leaving
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, prefill_tc_kernel<D>, tp);
}

}  // namespace

cudaError_t launch_prefill_tc(const PrefillParams &p, int head_dim, int cover, cudaStream_t stream) {
  PfTcParams tp = {};
  tp.p = p;
  tp.cover = cover;
  tp.n_qt = (cover + kTcTok - 1) / kTcTok;
  const long long rows = (long long)p.num_pages * p.n_kvh * p.page_size;
  if (!pool_tensor_map(&tp.tmap_k, p.k_pages, rows, head_dim, false) ||
      !pool_tensor_map(&tp.tmap_v, p.v_pages, rows, head_dim, false))
    return cudaErrorInvalidValue;
  return head_dim == 64 ? launch_tc_t<64>(tp, stream) : launch_tc_t<128>(tp, stream);
}

}  // namespace kvattn
