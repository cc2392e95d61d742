// Long-prompt prefill attention on the fifth-generation tensor cores
// (tcgen05): the FlashAttention-2 blocking of "Qwen3-8B inference engine from
// scratch in C++/CUDA", section 4.4.1 (key blocks, a running maximum and
// normaliser per row, never the whole score matrix), with the causal mask of
// "LLM inference from smollm3.go", section "Prefill: the whole prompt at once"
// (new token i of a sequence attends over keys 0 .. ctx + i).
//
// A CTA owns 64 new tokens of one sequence x the 4 query heads of one group:
// two halves of 128 MMA rows (row 32 hh + tl of half hf: head hh of the group,
// token 32 hf + tl), so every staged K/V tile serves the whole group (section
// 4.4.2 of the Qwen3-8B page) and both halves.  Keys come in tiles of 128.
// Eleven warps:
//   * warps 0-3 (half 0) and 4-7 (half 1), one thread per row, TMEM lanes
//     32 (w % 4) .. of the half's 256 columns (S and P in 0-127, O in 128-):
//     per tile read the row's 128 scores S from tensor memory, mask them,
//     keep the running maximum m and normaliser l (log2 units; the maximum
//     moves lazily, by more than 8, so the accumulator is rarely rescaled),
//     and write
//     P = 2^(S - m) as bf16 pairs back over S in tensor memory; at the end
//     read O, divide by l, store bf16 (or the partial state of a split);
//   * warps 8 and 9: TMA tensor copies of the query rows (which the append
//     kernel rotated, scaled and left in the output rows) and the K tiles,
//     and of the V tiles (16-key page blocks, [16 rows][128 bytes] boxes,
//     128-byte swizzle) into a K ring and a V ring of 2 (d 128) or 3 (d 64)
//     slots; a thread issues about one copy every 115 clocks, so each ring
//     has its own issuer;
//   * warp 10, one thread: issues the MMAs and commits them to mbarriers:
//     S = Q K^T (M 128, N 128, K d; both operands in shared memory) and
//     O += P V (M 128, N d, K 128; P from tensor memory, V in shared memory).
// N of 128 keeps the tensor pipe at its rate with operands read from shared
// memory (at N 64 the reads of A bound it), and P never passes through shared
// memory.  Per half the steps are serial (S(i + 1) overwrites P(i) once the
// P V products of tile i are done); the two halves interleave, so one half's
// MMAs run while the other's softmax works.  Every wait is bounded
// (KVATTN_DEV_TIMEOUT).
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <mutex>

#include "prefill_common.cuh"

namespace kvattn {

namespace {

constexpr int kTcHalf = kTcTok / 2;  // new tokens of a half
constexpr int kTcRows = 4 * kTcHalf; // MMA M: 32 new tokens x 4 heads
constexpr int kTcSoftWarps = 8;      // two halves of four warps
// warps kTcSoftWarps, + 1: the K and the V producer (one thread issues a
// tensor copy every ~115 clocks, so the two rings get an issuer each);
// kTcSoftWarps + 2: the MMA issuer
constexpr int kTcThreads = 32 * (kTcSoftWarps + 3);
constexpr uint32_t kTmemCols = 512;  // per half: S / P in 128 columns, O in d
constexpr uint32_t kHalfCols = 256;
constexpr uint32_t kOCol = 128;      // O's first TMEM column in a half

template <int D>
struct TcCfg {
  static constexpr int kStages = D == 128 ? 2 : 3;           // K/V tiles in flight
  static constexpr int kRegions = D / 64;                    // 128-byte column blocks of a row
  static constexpr int kQRegion = kTcRows * 128;             // [128 rows][128 B]
  static constexpr int kQHalf = kRegions * kQRegion;         // a half's Q
  static constexpr int kKVRegion = kTcKeys * 128;            // [128 keys][128 B]
  static constexpr int kTile = kRegions * kKVRegion;         // K or V tile
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + 2 * kQHalf;            // K ring [kStages][kTile]
  static constexpr int kVOff = kKOff + kStages * kTile;       // V ring [kStages][kTile]
  static constexpr int kBarOff = kVOff + kStages * kTile;
  // k_full[S], v_full[S], k_empty[S], v_empty[S], s_full[2], p_full[2],
  // o_done[2], q_ready[2], mma_done, out_bar[2]
  static constexpr int kNumBars = 4 * kStages + 11;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;    // tmem base, abort flag, counters
  static constexpr int kSmem = kMiscOff + 64 + 1024;         // + slack for 1024-byte alignment
  static_assert(kSmem <= 227 * 1024, "shared memory");
  static_assert(kKOff % 1024 == 0 && kTile % 1024 == 0, "swizzle atoms need 1024-byte alignment");
};

struct PfTcParams {
  CUtensorMap tmap_k, tmap_v;  // [rows][D] bf16 pools, [16][64] boxes, 128-byte swizzle
  // [n_tok][n_qh][D] bf16 view of out, where the append kernel left the
  // rotated, scaled query rows: [32 tokens][1 head][64] boxes, 128-byte swizzle
  CUtensorMap tmap_q;
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
// (no memory clobber: the operands are ordered by the mbarrier waits and
// fences around the issue loop, and the address arithmetic may be scheduled
// ahead of the instruction)
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(acc));
}
// D (TMEM, fp32) = A B (+ D when acc): A bf16 in tensor memory (row r in lane
// r, two consecutive K elements a 32-bit column), B bf16 in shared memory
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                          uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(acc));
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


// Columns c .. c + 127 of this thread's TMEM lane as fp32, the wait in the
// same statement.
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, float (&v)[128]) {
  uint32_t r[128];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x128.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, %64, %65, %66, %67, %68, %69, %70, %71, %72, %73, %74, %75, %76, %77, %78, %79, %80, %81, %82, %83, %84, %85, %86, %87, %88, %89, %90, %91, %92, %93, %94, %95, %96, %97, %98, %99, %100, %101, %102, %103, %104, %105, %106, %107, %108, %109, %110, %111, %112, %113, %114, %115, %116, %117, %118, %119, %120, %121, %122, %123, %124, %125, %126, %127}, [%128];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
        "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
        "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]),
        "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]),
        "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]),
        "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]),
        "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]),
        "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]),
        "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]),
        "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]),
        "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 128; ++i) v[i] = __uint_as_float(r[i]);
}

// Store 64 raw 32-bit columns (bf16 pairs) of this thread's TMEM lane and
// wait for the stores to complete.
__device__ __forceinline__ void tmem_st64u(uint32_t taddr, const uint32_t (&v)[64]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, %64};\n\t"
      "tcgen05.wait::st.sync.aligned;"
      :
      : "r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]),
        "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]),
        "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31]),
        "r"(v[32]), "r"(v[33]), "r"(v[34]), "r"(v[35]), "r"(v[36]), "r"(v[37]), "r"(v[38]), "r"(v[39]),
        "r"(v[40]), "r"(v[41]), "r"(v[42]), "r"(v[43]), "r"(v[44]), "r"(v[45]), "r"(v[46]), "r"(v[47]),
        "r"(v[48]), "r"(v[49]), "r"(v[50]), "r"(v[51]), "r"(v[52]), "r"(v[53]), "r"(v[54]), "r"(v[55]),
        "r"(v[56]), "r"(v[57]), "r"(v[58]), "r"(v[59]), "r"(v[60]), "r"(v[61]), "r"(v[62]), "r"(v[63])
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

// 3-D TMA tensor store of a box in shared memory (bulk group completion)
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, const void *src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(z), "r"(smem_addr(src))
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// this thread's committed bulk stores have read their shared-memory sources
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// 3-D TMA tensor copy with the default L2 policy
__device__ __forceinline__ void tma_load_3d_keep(void *dst, const CUtensorMap *map, int x, int y, int z,
                                                 uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
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

// Largest of N values: a tree of three-input maxima (N / 2 instructions, no
// long chain of dependent ones)
template <int N>
__device__ __forceinline__ float max_of(const float (&s)[N]) {
  float t[(N + 2) / 3];
  constexpr int M = N / 3;
#pragma unroll
  for (int k = 0; k < M; ++k) t[k] = max3f(s[3 * k], s[3 * k + 1], s[3 * k + 2]);
  if constexpr (N % 3 == 1) t[M] = s[N - 1];
  if constexpr (N % 3 == 2) t[M] = fmaxf(s[N - 2], s[N - 1]);
  if constexpr ((N + 2) / 3 == 1) {
    return t[0];
  } else {
    return max_of<(N + 2) / 3>(t);
  }
}

template <int D>
__global__ void __launch_bounds__(kTcThreads, 1) prefill_tc_kernel(const __grid_constant__ PfTcParams tp) {
  using C = TcCfg<D>;
  constexpr int S = C::kStages;
  const PrefillParams &p = tp.p;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kBarOff);
  uint64_t *k_full = bars, *v_full = bars + S, *k_empty = bars + 2 * S, *v_empty = bars + 3 * S;
  uint64_t *s_full = bars + 4 * S;  // [half]
  uint64_t *p_full = s_full + 2;    // [half]
  uint64_t *o_done = p_full + 2;    // [half]
  uint64_t *q_ready = o_done + 2;  // [half]: its query rows have landed
  uint64_t *mma_done = q_ready + 2;
  uint64_t *out_bar = mma_done + 1;  // [half]: its output rows are in shared memory
  uint32_t *misc = reinterpret_cast<uint32_t *>(smem + C::kMiscOff);
  uint32_t *tmem_slot = misc;                                 // [0]
  volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + 1);
  volatile int *issued_k = reinterpret_cast<volatile int *>(misc + 2);
  volatile int *issued_v = reinterpret_cast<volatile int *>(misc + 3);
  uint8_t *qs = smem + C::kQOff;
  uint8_t *kring = smem + C::kKOff, *vring = smem + C::kVOff;

  // (initialised first, while the sequence's lengths load; a CTA that leaves
  // early never uses them)
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], kTcRows);
      mbar_init(&o_done[i], 1);
      mbar_init(&out_bar[i], kTcRows);
    }
    mbar_init(&q_ready[0], 1);
    mbar_init(&q_ready[1], 1);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    *issued_k = 0;
    *issued_v = 0;
    fence_barrier_init();
  }

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
    if (qt == 0 && grp == 0 && tid == 0 && blockIdx.z == 0) report(p, KVATTN_DEV_BAD_LEN);
    pdl_wait_primary();
    return;
  }
  if (qt == 0 && grp == 0 && tid == 0 && blockIdx.z == 0 && n_new > tp.cover)
    report(p, KVATTN_DEV_BAD_LEN);
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
  // The CTA visits its key tiles starting at a rotation of its own: the CTAs
  // of one sequence and head group that run at once (the query tiles of one
  // wave) would otherwise all copy tile 0, then tile 1, ... at the same time
  // and queue on the same L2 lines.  (The online softmax takes the tiles in
  // any order.)
  const int rot = n_tiles > 1 ? (int)(((unsigned)qt * 5u + (unsigned)grp) % (unsigned)n_tiles) : 0;
  const auto tile_at = [&](int i) { return kt0 + (i + rot < n_tiles ? i + rot : i + rot - n_tiles); };

  __syncthreads();  // the barriers are initialised
  // The tensor memory is allocated by warp 0 and its address shared with the
  // softmax and MMA warps by a named barrier: the producers, which do not use
  // it, start copying at once.
  constexpr int kTmemUsers = 32 * (kTcSoftWarps + 1);
  uint32_t tmem = 0;
  if (warp < kTcSoftWarps || warp == kTcSoftWarps + 2) {
    if (warp == 0) {
      tmem_alloc(tmem_slot, kTmemCols);
      tmem_relinquish();
    }
    tc_fence_before();
    asm volatile("bar.sync 1, %0;" ::"n"(kTmemUsers) : "memory");
    tc_fence_after();
    tmem = *tmem_slot;
  }

  if (warp < kTcSoftWarps) {
    // ---- softmax warps: one thread per row ------------------------------------
    const int hf = warp >> 2, wq = warp & 3;
    const int h = h0 + wq, t = t0 + kTcHalf * hf + lane;
    const bool live = t < n_rows_tok;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * wq) << 16) + kHalfCols * (uint32_t)hf;
    const int kmax = live ? ctx + t : -1;  // last key the row sees
    const float kFloor = -1e30f;
    float m_run = kFloor, l_run = 0.f;
    int i = 0;
    for (; i < n_tiles; ++i) {
      if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
      // masks: causal (key <= ctx + t), and pages outside the pool (lanes 0-7
      // look up the tile's eight 16-key blocks, before the scores are waited
      // for); a tile every row of the warp sees whole, on valid pages, needs none
      const int key0 = tile_at(i) * kTcKeys;
      int pg = 0;
      if (lane < kTcKeys / 16 && key0 + 16 * lane < n_keys)
        pg = __ldg(p.block_table + (size_t)b * p.max_pages + ((key0 + 16 * lane) >> p.page_shift));
      {
        // one lane polls for the scores, the warp follows it
        bool got = true;
        if (lane == 0) got = tc_wait(&s_full[hf], (uint32_t)(i & 1), abort_flag, p);
        if (!__shfl_sync(0xffffffffu, got, 0)) break;
      }
      tc_fence_after();
      // the row's 128 scores in one load
      float sc[kTcKeys];
      tmem_ld128(lane_base, sc);
      const unsigned vbits = __ballot_sync(0xffffffffu, pg >= 0 && pg < p.num_pages) & 0xFFu;
      if (__any_sync(0xffffffffu, key0 + kTcKeys - 1 > kmax) || vbits != 0xFFu) {
#pragma unroll
        for (int c = 0; c < kTcKeys; ++c) {
          const bool ok = ((vbits >> (c >> 4)) & 1u) && key0 + c <= kmax;
          sc[c] = ok ? sc[c] : -INFINITY;
        }
      }
      const float m_new = fmaxf(m_run, max_of<kTcKeys>(sc));
      const bool need = m_new > m_run + 8.f;
      const float alpha = need ? ex2_approx(m_run - m_new) : 1.f;
      if (need) {
        m_run = m_new;
        l_run *= alpha;
      }
      // The last tile may end inside a 16-key block whose rows past the keys
      // hold whatever the pool has there (possibly not a number): half 0 zeroes
      // those V rows, so that their zero weights cannot meet a NaN in the MMA
      // (the masked scores are selected away, so stale K rows do no harm).
      // Both halves' products of the tile are issued after half 0's P.
      if (hf == 0 && tile_at(i) == all_tiles - 1 && (n_keys & 15) != 0) {
        const int st = i % S;
        if (!__all_sync(0xffffffffu, tc_wait(&v_full[st], (uint32_t)((i / S) & 1), abort_flag, p))) break;
        const int r0 = n_keys - key0, r1 = (r0 + 15) & ~15;
        uint8_t *vt = vring + st * C::kTile;
        for (int e = tid; e < (r1 - r0) * C::kRegions * 8; e += kTcRows) {
          const int r = r0 + e / (C::kRegions * 8), rr = e % (C::kRegions * 8);
          *reinterpret_cast<uint4 *>(vt + (rr >> 3) * C::kKVRegion + r * 128 + (rr & 7) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
      }
      // P = 2^(S - m) as bf16 pairs over the first 64 columns of S (column c:
      // keys 2c, 2c + 1), in one store; the differences and the normaliser's
      // sums two by two from packed fp32 arithmetic (one instruction a pair:
      // the chain of this loop is what a tile waits for), the sums in four
      // partial pairs.  fp32 exponentials: the f16 pair exponential takes half
      // the special-function operations but three conversions a pair more,
      // which made the chain longer (0.214 against 0.207 ms a prompt batch).
      float2 ls[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
      {
        uint32_t pw[kTcKeys / 2];
#pragma unroll
        for (int c = 0; c < kTcKeys / 2; ++c) {
          const float2 d = sub_f32x2(sc[2 * c], sc[2 * c + 1], m_run);
          const float2 e = make_float2(ex2_approx(d.x), ex2_approx(d.y));
          ls[c & 3] = add_f32x2(ls[c & 3], e);
          pw[c] = pack_bf16(e.x, e.y);
        }
        tmem_st64u(lane_base, pw);
      }
      l_run += ((ls[0].x + ls[0].y) + (ls[1].x + ls[1].y)) + ((ls[2].x + ls[2].y) + (ls[3].x + ls[3].y));
      // O holds the products of tiles < i, all complete: the MMA thread issued
      // S(i) only after them.  Rescale this warp's rows when a maximum moved.
      if (i > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          float o[32];
          tmem_ld32(lane_base + kOCol + (uint32_t)c0, o);
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] *= alpha;
          tmem_st32(lane_base + kOCol + (uint32_t)c0, o);
        }
      }
      tc_fence_before();
      mbar_arrive(&p_full[hf]);
    }
    // ---- the row's output: O / l rounded to bf16, or (several splits) the
    // partial state o (relative to 2^m), m, l for the merge kernel ------------
    if (i == n_tiles) {
      const int last = n_tiles - 1;
      const bool ok = n_tiles == 0 ||
                      __all_sync(0xffffffffu, tc_wait(&o_done[hf], (uint32_t)(last & 1), abort_flag, p));
      if (ok) {
        if (n_tiles > 0) tc_fence_after();
        const float f = l_run > 0.f ? 1.f / l_run : 0.f;  // no visible key: a zero row
        __nv_bfloat16 *dst = p.out + ((size_t)(start + (live ? t : 0)) * p.n_qh + h) * D;
        float *rec = p.part + (((size_t)z * p.n_tok + start + (live ? t : 0)) * p.n_qh + h) * (D + 2);
        const bool split = p.n_splits > 1;
        // A half whose 32 tokens are all this sequence's new rows (so a whole
        // box is the CTA's own) leaves its bf16 rows in shared memory, where
        // its query rows were (the last scores are complete), in the query
        // copies' swizzled layout, and one thread writes them out with the
        // same tensor map: whole lines instead of each thread's 16-byte pieces
        // of rows 4 KB apart.
        const bool boxed = !split && n_tiles > 0 && t0 + kTcHalf * (hf + 1) <= n_rows_tok;
        if (boxed) {
          uint8_t *qrow = qs + hf * C::kQHalf + wq * (kTcHalf * 128) + lane * 128;
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 32) {
            float o[32];
            tmem_ld32(lane_base + kOCol + (uint32_t)c0, o);
#pragma unroll
            for (int k = 0; k < 32; k += 8) {
              const int c = (c0 + k) / 8;  // 16-byte chunk of the row: block c / 8, chunk c % 8 in it
              const uint4 v = make_uint4(pack_bf16(o[k] * f, o[k + 1] * f), pack_bf16(o[k + 2] * f, o[k + 3] * f),
                                         pack_bf16(o[k + 4] * f, o[k + 5] * f), pack_bf16(o[k + 6] * f, o[k + 7] * f));
              *reinterpret_cast<uint4 *>(qrow + (c >> 3) * C::kQRegion + (((c & 7) ^ (lane & 7)) << 4)) = v;
            }
          }
          fence_proxy_async_smem();
          mbar_arrive(&out_bar[hf]);  // (release: the row is visible)
          if (wq == 0 && lane == 0 && tc_wait(&out_bar[hf], 0, abort_flag, p)) {
#pragma unroll
            for (int hh = 0; hh < 4; ++hh)
#pragma unroll
              for (int r = 0; r < C::kRegions; ++r)
                tma_store_3d(&tp.tmap_q, qs + hf * C::kQHalf + r * C::kQRegion + hh * (kTcHalf * 128), 64 * r,
                             h0 + hh, start + t0 + kTcHalf * hf);
            bulk_commit();
            bulk_wait_read_all();  // the rows are read before the shared memory is given up
          }
        }
#pragma unroll 1
        for (int c0 = 0; c0 < D && !boxed; c0 += 32) {
          float o[32];
          if (n_tiles > 0) {
            tmem_ld32(lane_base + kOCol + (uint32_t)c0, o);
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
  } else if (warp <= kTcSoftWarps + 1) {
    // ---- producers: the K tiles (warp 8) and the V tiles (warp 9) by TMA --------
    // K(i) and V(i) have rings of their own: K(i) is released once both halves'
    // scores of tile i are done, V(i) once their P V products are, so the
    // next keys start loading well before the weighted sums end
    const bool is_v = warp == kTcSoftWarps + 1;
    prefetch_tensormap(is_v ? &tp.tmap_v : &tp.tmap_k);
    // pool row of each 16-key block of tile i (lanes 0-7); rows past the keys
    // or on an out-of-range page are fetched from row -16, outside the view,
    // which the copy fills with zeros (the block table is no output of the
    // append grid: the first tile's rows are found before the wait on it)
    auto pool_rows = [&](int i) {
      int prow = -16;
      if (lane < kTcKeys / 16) {
        const int key = tile_at(i) * kTcKeys + 16 * lane;
        if (key < n_keys) {
          const int pg = __ldg(p.block_table + (size_t)b * p.max_pages + (key >> p.page_shift));
          if (pg >= 0 && pg < p.num_pages)
            prow = (pg * p.n_kvh + j) * p.page_size + (key & (p.page_size - 1));
          else if (!is_v)
            report(p, KVATTN_DEV_BAD_PAGE);
        }
      }
      return prow;
    };
    const int prow0 = n_tiles > 0 ? pool_rows(0) : -16;
    pdl_wait_primary();  // the appended rows and the query rows are complete and visible
    uint64_t *ring_full = is_v ? v_full : k_full, *ring_empty = is_v ? v_empty : k_empty;
    uint8_t *ring = is_v ? vring : kring;
    volatile int *issued = is_v ? issued_v : issued_k;
    const CUtensorMap *map = is_v ? &tp.tmap_v : &tp.tmap_k;
    auto wait_slot = [&](uint64_t *bar, uint32_t parity) -> bool {
      bool ok = true;
      if (lane == 0) ok = tc_wait(bar, parity, abort_flag, p);
      return __shfl_sync(0xffffffffu, ok, 0);
    };
    for (int i = 0; i < n_tiles; ++i) {
      if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
      const int s = i % S;
      const int prow = i == 0 ? prow0 : pool_rows(i);
      int rows[kTcKeys / 16];
#pragma unroll
      for (int q8 = 0; q8 < kTcKeys / 16; ++q8) rows[q8] = __shfl_sync(0xffffffffu, prow, q8);
      if (i >= S && !wait_slot(&ring_empty[s], (uint32_t)(((i / S) - 1) & 1))) break;
      if (lane == 0) {
        uint8_t *dst = ring + s * C::kTile;
        mbar_arrive_expect_tx(&ring_full[s], C::kTile);
#pragma unroll
        for (int q8 = 0; q8 < kTcKeys / 16; ++q8)
#pragma unroll
          for (int r = 0; r < C::kRegions; ++r)
            tma_load_2d_keep(dst + r * C::kKVRegion + q8 * 2048, map, 64 * r, rows[q8], &ring_full[s]);
        *issued = i + 1;
      }
      __syncwarp();
    }
  } else {
    // ---- MMA issuer: one thread -------------------------------------------------------
    pdl_wait_primary();
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16(kTcRows, kTcKeys, false);
      constexpr uint32_t kIdPV = idesc_bf16(kTcRows, D, true);
      // Descriptors of the first operand blocks, formed once: every other
      // block (k-step, stage, half) is a constant number of 16-byte units on,
      // added to the start-address field (which never carries: shared
      // addresses stay below 2^18)
      const uint32_t q0 = smem_addr(qs);
      const uint64_t dq = sw128_desc(q0, 16, 1024);               // Q, K-major
      const uint64_t dk = sw128_desc(smem_addr(kring), 16, 1024);  // K tiles, K-major
      // V tiles, MN-major: rows of 64 d (one 128-byte swizzle atom across),
      // 8-key groups 1024 bytes apart, the next 64 d one region on
      const uint64_t dv = sw128_desc(smem_addr(vring), C::kKVRegion, 1024);
      // both halves' query rows, issued here so that the K producer's first
      // tile goes out at the same time: a [32 tokens][64] box per head and
      // 64-column block, rows 32 hh + tl of the half's tile (tokens past the
      // new rows are another sequence's or, past n_tok, zeros: never stored)
      // (a barrier a half: half 0's first scores need only its own rows)
      prefetch_tensormap(&tp.tmap_q);
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        mbar_arrive_expect_tx(&q_ready[hf], C::kQHalf);
#pragma unroll
        for (int hh = 0; hh < 4; ++hh)
#pragma unroll
          for (int r = 0; r < C::kRegions; ++r)
            tma_load_3d_keep(qs + hf * C::kQHalf + r * C::kQRegion + hh * (kTcHalf * 128), &tp.tmap_q, 64 * r,
                             h0 + hh, start + t0 + kTcHalf * hf, &q_ready[hf]);
      }
      bool ok = true;
      auto issue_s = [&](int i, int hf) {
        const int s = i % S;
        const uint64_t kst = dk + (uint64_t)((s * C::kTile) >> 4);
        const uint64_t qh = dq + (uint64_t)((hf * C::kQHalf) >> 4);
        const uint32_t d_s = tmem + kHalfCols * (uint32_t)hf;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          // k-step ks: 64-element column block ks / 4, 32 bytes per step inside it
          const uint64_t oq = (uint64_t)(((ks >> 2) * C::kQRegion + (ks & 3) * 32) >> 4);
          const uint64_t ok2 = (uint64_t)(((ks >> 2) * C::kKVRegion + (ks & 3) * 32) >> 4);
          tc_mma(d_s, qh + oq, kst + ok2, kIdS, ks > 0 ? 1u : 0u);
        }
        tc_commit(&s_full[hf]);
      };
      auto issue_pv = [&](int i, int hf) {
        const int s = i % S;
        const uint64_t vst = dv + (uint64_t)((s * C::kTile) >> 4);
        const uint32_t d_o = tmem + kHalfCols * (uint32_t)hf + kOCol;
        const uint32_t a_p = tmem + kHalfCols * (uint32_t)hf;  // P: columns 0-63 of the half
        const uint32_t acc0 = i > 0 ? 1u : 0u;
#pragma unroll
        for (int ks = 0; ks < kTcKeys / 16; ++ks)
          // 16 keys: 8 columns of P; two 8-row groups = 2048 bytes of V on
          tc_mma_ts(d_o, a_p + (uint32_t)(8 * ks), vst + (uint64_t)(ks * 128), kIdPV, ks > 0 ? 1u : acc0);
        tc_commit(&o_done[hf]);
      };
      // Per tile, half by half: P V(i) of the half once its P(i) is written
      // (and V(i) has landed), then its S(i + 1) once that P V(i) is done
      // (S(i + 1) overwrites P(i)) and K(i + 1) has landed.  So a half's next
      // scores never wait for the other half's weights: while one half's
      // softmax works, the tensor pipe runs the other half's products
      // (ping-pong).
      if (n_tiles > 0) {
        ok = tc_wait(&q_ready[0], 0, abort_flag, p) && tc_wait(&k_full[0], 0, abort_flag, p);
        if (ok) {
          tc_fence_after();
          issue_s(0, 0);
          ok = tc_wait(&q_ready[1], 0, abort_flag, p);
        }
        if (ok) {
          tc_fence_after();
          issue_s(0, 1);
          tc_commit(&k_empty[0]);  // both halves' scores of tile 0 issued
        }
      } else {
        // (no tiles: the query copies land before the CTA leaves)
        ok = tc_wait(&q_ready[0], 0, abort_flag, p) && tc_wait(&q_ready[1], 0, abort_flag, p);
      }
      for (int i = 0; ok && i < n_tiles; ++i) {
        if (*abort_flag) break;
        const int s = i % S, s1 = (i + 1) % S;
        const bool more = i + 1 < n_tiles;
        ok = tc_wait(&v_full[s], (uint32_t)((i / S) & 1), abort_flag, p);
        for (int hf = 0; hf < 2 && ok; ++hf) {
          ok = tc_wait(&p_full[hf], (uint32_t)(i & 1), abort_flag, p);
          if (!ok) break;
          tc_fence_after();
          issue_pv(i, hf);
          if (hf == 1) tc_commit(&v_empty[s]);  // both halves' P V(i) issued
          if (!more) continue;
          if (hf == 0) ok = tc_wait(&k_full[s1], (uint32_t)(((i + 1) / S) & 1), abort_flag, p);
          if (ok) ok = tc_wait(&o_done[hf], (uint32_t)(i & 1), abort_flag, p);
          if (!ok) break;
          tc_fence_after();
          issue_s(i + 1, hf);
          if (hf == 1) tc_commit(&k_empty[s1]);  // both halves' S(i + 1) issued
        }
      }
      // every MMA issued has completed before the tensor memory is freed
      tc_commit(mma_done);
      (void)tc_wait(mma_done, 0, abort_flag, p);
    }
    __syncwarp();
  }

  __syncthreads();
  if (warp == kTcSoftWarps && lane == 0 && *abort_flag) {
    // copies still in flight on a slot nobody waited for land before the CTA leaves
    const int nk = *issued_k, nv = *issued_v;
    for (int i = max(0, nk - S); i < nk; ++i) (void)mbar_wait_bounded(&k_full[i % S], (uint32_t)((i / S) & 1));
    for (int i = max(0, nv - S); i < nv; ++i) (void)mbar_wait_bounded(&v_full[i % S], (uint32_t)((i / S) & 1));
    (void)mbar_wait_bounded(&q_ready[0], 0);
    (void)mbar_wait_bounded(&q_ready[1], 0);
  }
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// 3-D view [n_tok][n_qh][head_dim] of the bf16 rows at `base` in [32 tokens]
// [1 head][64 columns] boxes with 128-byte swizzle
bool query_tensor_map(CUtensorMap *map, const void *base, int n_tok, int n_qh, int head_dim) {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)n_qh, (cuuint64_t)n_tok};
  cuuint64_t strides[2] = {(cuuint64_t)head_dim * 2, (cuuint64_t)n_qh * head_dim * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)kTcHalf};
  cuuint32_t estride[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estride,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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
      !pool_tensor_map(&tp.tmap_v, p.v_pages, rows, head_dim, false) ||
      !query_tensor_map(&tp.tmap_q, p.out, p.n_tok, p.n_qh, head_dim))
    return cudaErrorInvalidValue;
  return head_dim == 64 ? launch_tc_t<64>(tp, stream) : launch_tc_t<128>(tp, stream);
}

}  // namespace kvattn
