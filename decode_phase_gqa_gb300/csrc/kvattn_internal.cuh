// Internal declarations of the decode-attention library: kernel parameter
// blocks, workspace layout and small sm_100-family PTX wrappers (mbarrier,
// bulk async copy, programmatic dependent launch).  Not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvattn.h"

namespace kvattn {

// Tokens per work unit.  A page of page_size tokens (a multiple of 16) is
// streamed as page_size / 16 units; each unit is one contiguous
// [16][head_dim] block of the [page][kv_head][slot][d] pool.
constexpr int kUnitRows = 16;
constexpr int kDecodeWarps = 4;
constexpr int kDecodeThreads = kDecodeWarps * 32;
// Most 16-token units (over all streams) a step's block tables may hold.
constexpr long long kMaxStepUnits = (1LL << 28) - 1;
// shared memory a decode CTA may use so that 3 fit on one SM (228 KB, with
// 1 KB reserved per CTA)
constexpr int kCtaSmemBudget = 75 * 1024;
// The decode grid pulls the whole block table into L2 at its start when the
// table spans at most this many 128-byte lines (1 MB).
constexpr long long kTablePrefetchLines = 8192;
// A bounded wait gives up after this many SM clocks (about one second).
constexpr long long kWaitCycles = 2000000000LL;
#ifdef KVATTN_TEST_STALL
// Test builds only (the macro is never defined in the library build): when a
// call finds kTestStallRequest set in its status word, every decode warp
// first waits, with this short limit (about a millisecond), on a barrier that
// nothing ever arrives at and that no copy is ever issued to, so the wait runs
// out, KVATTN_DEV_TIMEOUT is recorded and the kernel takes its give-up path.
constexpr long long kTestStallCycles = 2000000LL;
constexpr uint32_t kTestStallRequest = 0x80000000u;
#endif

// Query heads per CTA group: the largest of 4, 2, 1 dividing the GQA group.
inline int group_split(int g) { return (g % 4 == 0) ? 4 : (g % 2 == 0) ? 2 : 1; }

struct DecodeParams {
  // 2-D views [n_layers * num_pages * n_kvh * page_size rows][head_dim] of the
  // K and V pools (all layers), [16 rows][128 or 64 bytes] boxes, swizzled
  CUtensorMap tmap_k, tmap_v;
  const int32_t *block_table, *seq_lens, *positions;
  const __nv_bfloat16 *q, *k_new, *v_new;
  void *k_pages, *v_pages;      // written only in the new token's slot
  float *k_scales, *v_scales;
  __nv_bfloat16 *out;
  float *records;      // partial softmax states of split streams
  uint32_t *status;
  int n_seq, n_qh, n_kvh, page_size, max_pages, num_pages;
  int n_layers;        // layer caches decoded by the call (layer-major arrays,
                       // one pool of num_pages pages per layer); 1 for one layer
  int n_sub;           // query-head groups per KV head (G / GS)
  int n_shares;        // the unit list is cut into at most this many shares
  int unit_shift;      // log2(page_size / 16): units per page
  int stream_cost;     // weight of a stream's fixed costs in the work split
                       // (quarters of a unit's weight)
  int use_rope;        // rope_theta > 0
  uint32_t nope[KVATTN_MAX_LAYERS / 32];  // bit l: layer l has no RoPE
  float qscale;        // scale * log2(e): scores come out in log2 units
  // turns per position of rotation pair i, rope_theta^(-2i/d) / (2 pi), as an
  // fp32 head and remainder (host-computed in double)
  float2 turns[64];
  // rope_theta^(-2i/d) in double: the angles of the stored key
  double inv_freq[64];
};

// floats of one partial record (acc[gs][d], m[gs], l[gs]), padded so every
// record starts on a 16-byte boundary
__host__ __device__ inline constexpr int record_floats(int gs, int d) {
  return (gs * (d + 2) + 3) & ~3;
}

// ---- workspace layout ----------------------------------------------------
struct WorkspaceLayout {
  size_t status_off, records_off, total;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline WorkspaceLayout workspace_layout(int n_seq, int n_qh, int n_kvh, int d) {
  WorkspaceLayout w;
  const int g = n_qh / n_kvh;
  const int gs = group_split(g);
  const size_t streams = (size_t)n_seq * n_kvh * (g / gs);
  w.status_off = 0;
  w.records_off = 256;
  const size_t records = streams + KVATTN_MAX_SPLITS;
  w.total = align_up(w.records_off + records * (size_t)record_floats(gs, d) * sizeof(float), 256);
  return w;
}

// ---- launchers (one per translation unit) ----------------------------------
// Decode kernel of one (head_dim, group split) configuration: stores the
// resident CTAs per SM in *ctas_per_sm (when non-NULL) and launches the kernel
// with `grid` CTAs when `launch` is set.
cudaError_t launch_decode_bf16(const DecodeParams &p, int head_dim, int gs, int grid,
                               cudaStream_t stream, int *ctas_per_sm, bool launch);
cudaError_t launch_decode_int8(const DecodeParams &p, int head_dim, int gs, int grid,
                               cudaStream_t stream, int *ctas_per_sm, bool launch);
// the same for several layer caches (p.n_layers > 1)
cudaError_t launch_decode_bf16_layers(const DecodeParams &p, int head_dim, int gs, int grid,
                                      cudaStream_t stream, int *ctas_per_sm, bool launch);
cudaError_t launch_decode_int8_layers(const DecodeParams &p, int head_dim, int gs, int grid,
                                      cudaStream_t stream, int *ctas_per_sm, bool launch);
// Merge of the partial records of the streams the decode kernel's work split
// cut (sms = the GPU's SM count).
cudaError_t launch_combine(const DecodeParams &p, int head_dim, int gs, int n_warps, int sms,
                           cudaStream_t stream);

// Record `err` as this thread's last CUDA error (kvattn_last_cuda_error) and
// return KVATTN_ECUDA (kvattn_api.cu).
int cuda_fail(cudaError_t err);

// The host checks of kvattn_decode / kvattn_decode_layers (kvattn_api.cu):
// KVATTN_OK when the arguments may be launched on; queues nothing.
int decode_check(int n_layers, const void *q, const void *k_new, const void *v_new,
                 const void *k_pages, const void *v_pages, const int32_t *block_table,
                 const int32_t *seq_lens, const int32_t *positions, const void *out, int n_seq,
                 int n_qh, int n_kvh, int head_dim, int page_size, float rope_theta, float scale,
                 int kv_dtype, int max_pages_per_seq, int num_pages, const float *k_scales,
                 const float *v_scales, const void *workspace, size_t workspace_bytes,
                 int num_splits);

#ifdef __CUDACC__
// ---- device helpers ----------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of an mbarrier; false if it did not complete within
// `limit` SM clocks (the caller records KVATTN_DEV_TIMEOUT and stops using data).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  long long limit = kWaitCycles) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > limit) return false;
  }
  return true;
}

// One bulk (TMA) copy global -> shared, completing on `bar` with its byte count.
// Both addresses 16-byte aligned, bytes a multiple of 16.  The data is read
// once per step, so it is marked evict-first in L2.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void pdl_wait_primary() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Whether layer l's query and new key are rotated.
__device__ __forceinline__ bool layer_rope(const DecodeParams &p, int l) {
  return p.use_rope != 0 && ((p.nope[l >> 5] >> (l & 31)) & 1u) == 0;
}

// Number of 16-token units a sequence with L cached tokens spans (the new
// one included); 0 when the length is out of range.
__device__ __forceinline__ int units_of(int L, long long cap_tokens) {
  return (L >= 0 && (long long)L + 1 <= cap_tokens) ? (L + kUnitRows) / kUnitRows : 0;
}
#endif

}  // namespace kvattn
