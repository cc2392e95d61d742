// Host side of the C ABI declared in include/kvattn.h: argument checks (fail
// closed, nothing is launched on an error), workspace layout, the RoPE
// frequency table, the TMA descriptors of the pools and the two launches of
// one decode step on the caller's stream: the split-KV attention kernel (which
// also appends the new token) and, as its programmatic dependent, the merge of
// the streams its work split cut.  No host synchronisation except in
// kvattn_read_device_status.
#include <cudaTypedefs.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "kvattn_internal.cuh"

using namespace kvattn;

namespace {

// Weight of a stream's fixed costs in the work split, in quarters of a
// 16-token unit: the query set-up at the stream's start and the new token's
// stored row at its end (the correctly rounded cos/sin and, int8, the
// quantisation) take about as long as streaming this many units when every
// warp of the GPU streams.
constexpr int kStreamCostBf16 = 4;
constexpr int kStreamCostInt8 = 12;

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool supported_page(int page) {
  return page == 16 || page == 32 || page == 64 || page == 128 || page == 256;
}

// SM count of the current device (cached per device).
cudaError_t sm_count(int *out) {
  static std::mutex mu;
  static int cache[128] = {0};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
  if (cache[dev] == 0) {
    err = cudaDeviceGetAttribute(&cache[dev], cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
  }
  *out = cache[dev];
  return cudaSuccess;
}

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime
// (no link-time dependency on libcuda)
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 2-D view [rows][head_dim] of a K or V pool in [16 rows][128 bytes] boxes
// with 128-byte swizzle (bf16: 64 columns; int8, head_dim 128: 128 columns),
// or [16][64 bytes] boxes with 64-byte swizzle (int8, head_dim 64): the box's
// rows are written with their 16-byte chunks permuted, which the kernel's
// ldmatrix addressing undoes
bool encode_pool_map(CUtensorMap *map, const void *base, long long rows, int head_dim, bool int8) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const int esize = int8 ? 1 : 2;
  const int row_bytes = head_dim * esize;
  const int box_bytes = row_bytes < 128 ? row_bytes : 128;
  cuuint64_t dims[2] = {(cuuint64_t)head_dim, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  cuuint32_t box[2] = {(cuuint32_t)(box_bytes / esize), 16};
  cuuint32_t estride[2] = {1, 1};
  return enc(map, int8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
             const_cast<void *>(base), dims, strides, box, estride,
             CU_TENSOR_MAP_INTERLEAVE_NONE,
             box_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Small caches of per-call host work that only depends on a few arguments:
// the RoPE frequency tables (64 pow calls) per (rope_theta, head_dim) and the
// pools' tensor maps per (base, rows, head_dim, element type).  A call takes
// its entries by copy under the lock; misses replace entries round robin.
struct FreqEntry {
  uint32_t theta_bits;
  int head_dim;
  double inv_freq[64];
  float2 turns[64];
};
struct MapEntry {
  const void *base;
  long long rows;
  int head_dim;
  bool int8;
  CUtensorMap map;
};
std::mutex g_cache_mu;
FreqEntry g_freq[8];
int g_freq_n = 0, g_freq_next = 0;
MapEntry g_maps[16];
int g_maps_n = 0, g_maps_next = 0;

// frequency of rotation pair i: rope_theta^(-2i/d) in double, and the same in
// turns (/ 2 pi) as an fp32 head and remainder; zero without RoPE
void freq_tables(float rope_theta, int head_dim, double *inv_freq, float2 *turns) {
  uint32_t bits;
  std::memcpy(&bits, &rope_theta, 4);
  std::lock_guard<std::mutex> lock(g_cache_mu);
  for (int e = 0; e < g_freq_n; ++e)
    if (g_freq[e].theta_bits == bits && g_freq[e].head_dim == head_dim) {
      std::memcpy(inv_freq, g_freq[e].inv_freq, sizeof(g_freq[e].inv_freq));
      std::memcpy(turns, g_freq[e].turns, sizeof(g_freq[e].turns));
      return;
    }
  FreqEntry &f = g_freq[g_freq_next];
  g_freq_next = (g_freq_next + 1) % 8;
  if (g_freq_n < 8) ++g_freq_n;
  f.theta_bits = bits;
  f.head_dim = head_dim;
  const bool use_rope = rope_theta > 0.0f;
  for (int i = 0; i < 64; ++i)
    f.inv_freq[i] = (use_rope && i < head_dim / 2) ? std::pow((double)rope_theta, -(2.0 * i) / head_dim) : 0.0;
  for (int i = 0; i < 64; ++i) {
    const double g = f.inv_freq[i] * 0.15915494309189535;  // / (2 pi)
    const float hi = (float)g;
    f.turns[i] = make_float2(hi, (float)(g - (double)hi));
  }
  std::memcpy(inv_freq, f.inv_freq, sizeof(f.inv_freq));
  std::memcpy(turns, f.turns, sizeof(f.turns));
}

bool cached_pool_map(CUtensorMap *map, const void *base, long long rows, int head_dim, bool int8) {
  {
    std::lock_guard<std::mutex> lock(g_cache_mu);
    for (int e = 0; e < g_maps_n; ++e)
      if (g_maps[e].base == base && g_maps[e].rows == rows && g_maps[e].head_dim == head_dim &&
          g_maps[e].int8 == int8) {
        *map = g_maps[e].map;
        return true;
      }
  }
  if (!encode_pool_map(map, base, rows, head_dim, int8)) return false;
  std::lock_guard<std::mutex> lock(g_cache_mu);
  MapEntry &m = g_maps[g_maps_next];
  g_maps_next = (g_maps_next + 1) % 16;
  if (g_maps_n < 16) ++g_maps_n;
  m.base = base;
  m.rows = rows;
  m.head_dim = head_dim;
  m.int8 = int8;
  m.map = *map;
  return true;
}

cudaError_t decode_launcher(const DecodeParams &p, int head_dim, int gs, bool int8, int grid,
                            cudaStream_t stream, int *ctas_per_sm, bool launch) {
  return int8 ? launch_decode_int8(p, head_dim, gs, grid, stream, ctas_per_sm, launch)
              : launch_decode_bf16(p, head_dim, gs, grid, stream, ctas_per_sm, launch);
}

}  // namespace

namespace kvattn {
namespace {
thread_local int g_last_cuda_error = 0;
}
// Record the CUDA error behind a KVATTN_ECUDA return (kvattn_last_cuda_error)
// and return KVATTN_ECUDA.
int cuda_fail(cudaError_t err) {
  g_last_cuda_error = (int)(err == cudaSuccess ? cudaErrorUnknown : err);
  return KVATTN_ECUDA;
}

// the frequency tables for the prefill kernels (prefill.cu)
void rope_tables(float rope_theta, int head_dim, double *inv_freq, float2 *turns) {
  freq_tables(rope_theta, head_dim, inv_freq, turns);
}
// the pools' TMA view for the tcgen05 prefill kernel (prefill_tc.cu)
bool pool_tensor_map(CUtensorMap *map, const void *base, long long rows, int head_dim, bool int8) {
  return cached_pool_map(map, base, rows, head_dim, int8);
}
}  // namespace kvattn

namespace kvattn {
// The host checks of a decode call (sizes, pointers, alignment, workspace),
// in the order decode_call makes them; KVATTN_OK when a launch may follow.
// Queues nothing.
int decode_check(int n_layers, const void *q, const void *k_new, const void *v_new,
                 const void *k_pages, const void *v_pages, const int32_t *block_table,
                 const int32_t *seq_lens, const int32_t *positions, const void *out, int n_seq,
                 int n_qh, int n_kvh, int head_dim, int page_size, float rope_theta, float scale,
                 int kv_dtype, int max_pages_per_seq, int num_pages, const float *k_scales,
                 const float *v_scales, const void *workspace, size_t workspace_bytes,
                 int num_splits) {
  // ---- shape checks ----
  if (n_layers < 1 || n_seq < 0 || n_qh < 1 || n_kvh < 1 || n_qh % n_kvh != 0 ||
      max_pages_per_seq < 1 || num_pages < 1 || num_splits < 0 || num_splits > KVATTN_MAX_SPLITS)
    return KVATTN_EINVAL;
  if (n_layers > KVATTN_MAX_LAYERS) return KVATTN_EUNSUPPORTED;
  if (!std::isfinite(scale) || std::isnan(rope_theta) || std::isinf(rope_theta))
    return KVATTN_EINVAL;
  if (head_dim != 64 && head_dim != 128) return KVATTN_EUNSUPPORTED;
  if (!supported_page(page_size)) return KVATTN_EUNSUPPORTED;
  if (kv_dtype != KVATTN_KV_BF16 && kv_dtype != KVATTN_KV_INT8) return KVATTN_EUNSUPPORTED;
  if (n_seq > KVATTN_MAX_SEQS || n_qh > 1024) return KVATTN_EUNSUPPORTED;
  if ((long long)max_pages_per_seq * page_size > (long long)INT_MAX) return KVATTN_EUNSUPPORTED;
  // pool rows (all layers) are addressed with 32-bit TMA coordinates
  if ((long long)n_layers * num_pages * n_kvh * page_size > (long long)INT_MAX)
    return KVATTN_EUNSUPPORTED;
  // the work split weighs the 16-token units of all streams in 32-bit integers
  {
    const long long streams =
        (long long)n_layers * n_seq * n_kvh * (n_qh / n_kvh / group_split(n_qh / n_kvh));
    const long long units = streams * ((long long)max_pages_per_seq * page_size / kUnitRows);
    if (units > kMaxStepUnits ||
        4 * units + streams * std::max(kStreamCostBf16, kStreamCostInt8) > (long long)INT_MAX)
      return KVATTN_EUNSUPPORTED;
  }
  const bool int8 = kv_dtype == KVATTN_KV_INT8;
  if (n_seq == 0) return KVATTN_OK;  // empty batch: nothing to read or write
  // ---- pointer checks ----
  if (!q || !k_new || !v_new || !k_pages || !v_pages || !block_table || !seq_lens ||
      !positions || !out)
    return KVATTN_EINVAL;
  if (!aligned(k_pages, 16) || !aligned(v_pages, 16) || !aligned(q, 16) || !aligned(k_new, 2) ||
      !aligned(v_new, 2) || !aligned(out, 2) || !aligned(block_table, 4) ||
      !aligned(seq_lens, 4) || !aligned(positions, 4))
    return KVATTN_EINVAL;
  if (int8 && (!k_scales || !v_scales || !aligned(k_scales, 16) || !aligned(v_scales, 16)))
    return KVATTN_EINVAL;
  const WorkspaceLayout wl = workspace_layout(n_layers * n_seq, n_qh, n_kvh, head_dim);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < wl.total)
    return KVATTN_EWORKSPACE;
  return KVATTN_OK;
}
}  // namespace kvattn

// One decode step over n_layers layer caches (layer-major arrays sharing the
// block table, lengths and positions); kvattn_decode is n_layers = 1.
static int decode_call(int n_layers, const void *q, const void *k_new, const void *v_new,
                       void *k_pages, void *v_pages, const int32_t *block_table,
                       const int32_t *seq_lens, const int32_t *positions, void *out, int n_seq,
                       int n_qh, int n_kvh, int head_dim, int page_size, float rope_theta,
                       float scale, int kv_dtype, void *stream, int max_pages_per_seq,
                       int num_pages, float *k_scales, float *v_scales, void *workspace,
                       size_t workspace_bytes, int num_splits, const uint8_t *layer_rope) {
  {
    const int rc = decode_check(n_layers, q, k_new, v_new, k_pages, v_pages, block_table,
                                seq_lens, positions, out, n_seq, n_qh, n_kvh, head_dim,
                                page_size, rope_theta, scale, kv_dtype, max_pages_per_seq,
                                num_pages, k_scales, v_scales, workspace, workspace_bytes,
                                num_splits);
    if (rc != KVATTN_OK || n_seq == 0) return rc;
  }
  const bool int8 = kv_dtype == KVATTN_KV_INT8;
  const WorkspaceLayout wl = workspace_layout(n_layers * n_seq, n_qh, n_kvh, head_dim);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int g = n_qh / n_kvh;
  const int gs = group_split(g);

  // ---- launch 1: append of the new token and split-KV attention ----
  const bool use_rope = rope_theta > 0.0f;
  DecodeParams dp = {};
  dp.block_table = block_table;
  dp.seq_lens = seq_lens;
  dp.positions = positions;
  dp.q = static_cast<const __nv_bfloat16 *>(q);
  dp.k_new = static_cast<const __nv_bfloat16 *>(k_new);
  dp.v_new = static_cast<const __nv_bfloat16 *>(v_new);
  dp.k_pages = k_pages;
  dp.v_pages = v_pages;
  dp.k_scales = k_scales;
  dp.v_scales = v_scales;
  dp.out = static_cast<__nv_bfloat16 *>(out);
  dp.records = reinterpret_cast<float *>(ws + wl.records_off);
  dp.status = reinterpret_cast<uint32_t *>(ws + wl.status_off);
  dp.use_rope = use_rope ? 1 : 0;
  // layers whose entry of layer_rope is 0 skip RoPE (a NoPE layer)
  if (layer_rope)
    for (int l = 0; l < n_layers; ++l)
      if (!layer_rope[l]) dp.nope[l >> 5] |= 1u << (l & 31);
  // scores are formed in log2 units: fold scale * log2(e) into the query
  dp.qscale = (float)((double)scale * 1.4426950408889634);
  freq_tables(rope_theta, head_dim, dp.inv_freq, dp.turns);
  dp.n_seq = n_seq;
  dp.n_qh = n_qh;
  dp.n_kvh = n_kvh;
  dp.page_size = page_size;
  dp.max_pages = max_pages_per_seq;
  dp.num_pages = num_pages;
  dp.n_layers = n_layers;
  dp.n_sub = g / gs;
  for (int u = page_size / kUnitRows; u > 1; u >>= 1) ++dp.unit_shift;
  dp.stream_cost = int8 ? kStreamCostInt8 : kStreamCostBf16;
  {
    const long long rows = (long long)n_layers * num_pages * n_kvh * page_size;
    if (!cached_pool_map(&dp.tmap_k, k_pages, rows, head_dim, int8) ||
        !cached_pool_map(&dp.tmap_v, v_pages, rows, head_dim, int8))
      return cuda_fail(cudaErrorInvalidValue);  // the tensor map could not be encoded
  }
  // the first call for a configuration on a device sets the kernel's shared
  // memory limit and caches its occupancy; later calls only launch.  A share
  // of the unit list is one warp's work.
  int sms = 0, per_sm = 0;
  cudaError_t err = sm_count(&sms);
  if (err != cudaSuccess) return cuda_fail(err);
  err = decode_launcher(dp, head_dim, gs, int8, 0, st, &per_sm, false);
  if (err != cudaSuccess) return cuda_fail(err);
  int shares = num_splits;
  if (shares == 0) shares = sms * (per_sm > 0 ? per_sm : 1) * kDecodeWarps;
  if (shares > KVATTN_MAX_SPLITS) shares = KVATTN_MAX_SPLITS;
  dp.n_shares = shares;
  const int grid = (shares + kDecodeWarps - 1) / kDecodeWarps;
  err = decode_launcher(dp, head_dim, gs, int8, grid, st, nullptr, true);
  if (err != cudaSuccess) return cuda_fail(err);
  // ---- launch 2: merge of the streams the warp shares split ----
  err = launch_combine(dp, head_dim, gs, shares, sms, st);
  if (err != cudaSuccess) return cuda_fail(err);
  return KVATTN_OK;
}

extern "C" {

size_t kvattn_workspace_size_layers(int n_layers, int n_seq, int n_qh, int n_kvh, int head_dim) {
  if (n_layers < 1 || n_layers > KVATTN_MAX_LAYERS || n_seq < 0 || n_seq > KVATTN_MAX_SEQS ||
      n_qh < 1 || n_kvh < 1 || n_qh % n_kvh != 0 || (head_dim != 64 && head_dim != 128))
    return 0;
  return workspace_layout(n_layers * n_seq, n_qh, n_kvh, head_dim).total;
}

size_t kvattn_workspace_size(int n_seq, int n_qh, int n_kvh, int head_dim) {
  return kvattn_workspace_size_layers(1, n_seq, n_qh, n_kvh, head_dim);
}

int kvattn_workspace_init(void *workspace, size_t workspace_bytes, void *stream) {
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < 256) return KVATTN_EWORKSPACE;
  const cudaError_t err =
      cudaMemsetAsync(workspace, 0, workspace_bytes, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? KVATTN_OK : cuda_fail(err);
}

int kvattn_decode_splits(const void *q, const void *k_new, const void *v_new, void *k_pages,
                         void *v_pages, const int32_t *block_table, const int32_t *seq_lens,
                         const int32_t *positions, void *out, int n_seq, int n_qh, int n_kvh,
                         int head_dim, int page_size, float rope_theta, float scale,
                         int kv_dtype, void *stream, int max_pages_per_seq, int num_pages,
                         float *k_scales, float *v_scales, void *workspace,
                         size_t workspace_bytes, int num_splits) {
  return decode_call(1, q, k_new, v_new, k_pages, v_pages, block_table, seq_lens, positions, out,
                     n_seq, n_qh, n_kvh, head_dim, page_size, rope_theta, scale, kv_dtype, stream,
                     max_pages_per_seq, num_pages, k_scales, v_scales, workspace, workspace_bytes,
                     num_splits, nullptr);
}

int kvattn_decode_layers(int n_layers, const void *q, const void *k_new, const void *v_new,
                         void *k_pages, void *v_pages, const int32_t *block_table,
                         const int32_t *seq_lens, const int32_t *positions, void *out, int n_seq,
                         int n_qh, int n_kvh, int head_dim, int page_size, float rope_theta,
                         float scale, int kv_dtype, void *stream, int max_pages_per_seq,
                         int num_pages, float *k_scales, float *v_scales, void *workspace,
                         size_t workspace_bytes, const uint8_t *layer_rope) {
  return decode_call(n_layers, q, k_new, v_new, k_pages, v_pages, block_table, seq_lens,
                     positions, out, n_seq, n_qh, n_kvh, head_dim, page_size, rope_theta, scale,
                     kv_dtype, stream, max_pages_per_seq, num_pages, k_scales, v_scales,
                     workspace, workspace_bytes, 0, layer_rope);
}

int kvattn_decode(const void *q, const void *k_new, const void *v_new, void *k_pages,
                  void *v_pages, const int32_t *block_table, const int32_t *seq_lens,
                  const int32_t *positions, void *out, int n_seq, int n_qh, int n_kvh,
                  int head_dim, int page_size, float rope_theta, float scale, int kv_dtype,
                  void *stream, int max_pages_per_seq, int num_pages, float *k_scales,
                  float *v_scales, void *workspace, size_t workspace_bytes) {
  return kvattn_decode_splits(q, k_new, v_new, k_pages, v_pages, block_table, seq_lens,
                              positions, out, n_seq, n_qh, n_kvh, head_dim, page_size,
                              rope_theta, scale, kv_dtype, stream, max_pages_per_seq, num_pages,
                              k_scales, v_scales, workspace, workspace_bytes, 0);
}

int kvattn_read_device_status(void *workspace, void *stream, uint32_t *bits) {
  if (!bits) return KVATTN_EINVAL;
  if (!workspace || !aligned(workspace, 256)) return KVATTN_EWORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t host = 0;
  cudaError_t err = cudaMemcpyAsync(&host, workspace, sizeof host, cudaMemcpyDeviceToHost, st);
  if (err == cudaSuccess) err = cudaStreamSynchronize(st);
  if (err == cudaSuccess) err = cudaMemsetAsync(workspace, 0, sizeof host, st);
  if (err == cudaSuccess) err = cudaStreamSynchronize(st);
  if (err != cudaSuccess) return cuda_fail(err);
  *bits = host;
  return KVATTN_OK;
}

const char *kvattn_status_string(int status) {
  switch (status) {
    case KVATTN_OK: return "ok";
    case KVATTN_EINVAL: return "invalid argument (null/misaligned pointer or inconsistent size)";
    case KVATTN_EUNSUPPORTED: return "unsupported head_dim, page_size, kv_dtype or size";
    case KVATTN_ECUDA: return "CUDA runtime error";
    case KVATTN_EWORKSPACE: return "workspace missing, misaligned or too small";
    default: return "unknown status";
  }
}

int kvattn_version(void) { return 101; }

int kvattn_last_cuda_error(void) { return g_last_cuda_error; }

}  // extern "C"
