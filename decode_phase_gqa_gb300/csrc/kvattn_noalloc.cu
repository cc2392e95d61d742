// kvattn_decode_noalloc: the decode step for callers that cannot provide a
// workspace and cannot let the library allocate one.
//
// Some callers have no way to obtain device memory at call time: a serving
// engine that reserved nearly all of HBM for its KV-page pool at start-up and
// keeps no allocator for anything else, or a plugin inside a host framework
// that owns every device allocation and does not allow plugins to call
// cudaMalloc.  For them the step's scratch (status word, partial softmax
// states) lives in one fixed array compiled into this library instead of in a
// caller-owned workspace.
//
// The array is a file-scope __device__ variable.  In host code its name only
// stands in for the symbol, it is not a device address, so the address is
// looked up with cudaGetSymbolAddress once per device (with that device
// current) and that address is what the kernels receive.  The looked-up
// address is kept for the life of the process: after cudaDeviceReset (or
// anything else that destroys and re-creates the device's primary context)
// the array may sit elsewhere, so this entry point must not be used across
// such a reset.
#include <mutex>

#include "kvattn_internal.cuh"

namespace {

// Every GPU that loads this library holds these bytes until the process exits.
__device__ __align__(256) unsigned char g_noalloc_scratch[KVATTN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 128;
std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device, looked up on the
// first call made with that device current.
cudaError_t scratch_address(void **out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void *p = nullptr;
    err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (err != cudaSuccess) return err;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" int kvattn_decode_noalloc(const void *q, const void *k_new, const void *v_new,
                                     void *k_pages, void *v_pages, const int32_t *block_table,
                                     const int32_t *seq_lens, const int32_t *positions,
                                     void *out, int n_seq, int n_qh, int n_kvh, int head_dim,
                                     int page_size, float rope_theta, float scale, int kv_dtype,
                                     void *stream, int max_pages_per_seq, int num_pages,
                                     float *k_scales, float *v_scales, uint32_t *dev_status) {
  const size_t need = kvattn_workspace_size(n_seq, n_qh, n_kvh, head_dim);
  if (need == 0 || n_seq == 0) {
    // invalid sizes (reported by the regular checks) or nothing to do
    return kvattn_decode(q, k_new, v_new, k_pages, v_pages, block_table, seq_lens, positions,
                         out, n_seq, n_qh, n_kvh, head_dim, page_size, rope_theta, scale,
                         kv_dtype, stream, max_pages_per_seq, num_pages, k_scales, v_scales,
                         nullptr, 0);
  }
  if (need > KVATTN_NOALLOC_SCRATCH_BYTES) return KVATTN_EUNSUPPORTED;
  if (dev_status && (reinterpret_cast<uintptr_t>(dev_status) % 4) != 0) return KVATTN_EINVAL;
  void *scratch = nullptr;
  {
    const cudaError_t err = scratch_address(&scratch);
    if (err != cudaSuccess) return kvattn::cuda_fail(err);
  }
  // every host check of the decode step first, so that a rejected call has
  // queued nothing (not even the status clear below)
  {
    const int rc = kvattn::decode_check(1, q, k_new, v_new, k_pages, v_pages, block_table,
                                        seq_lens, positions, out, n_seq, n_qh, n_kvh, head_dim,
                                        page_size, rope_theta, scale, kv_dtype,
                                        max_pages_per_seq, num_pages, k_scales, v_scales,
                                        scratch, KVATTN_NOALLOC_SCRATCH_BYTES, 0);
    if (rc != KVATTN_OK) return rc;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the array keeps the previous call's contents: the status word must start
  // at zero (every record the combine kernel reads is rewritten by the step)
  {
    const cudaError_t err = cudaMemsetAsync(scratch, 0, 256, st);
    if (err != cudaSuccess) return kvattn::cuda_fail(err);
  }
  const int rc = kvattn_decode(q, k_new, v_new, k_pages, v_pages, block_table, seq_lens,
                               positions, out, n_seq, n_qh, n_kvh, head_dim, page_size,
                               rope_theta, scale, kv_dtype, stream, max_pages_per_seq, num_pages,
                               k_scales, v_scales, scratch, KVATTN_NOALLOC_SCRATCH_BYTES);
  if (rc != KVATTN_OK) return rc;
  if (dev_status) {
    const cudaError_t err =
        cudaMemcpyAsync(dev_status, scratch, sizeof(uint32_t), cudaMemcpyDeviceToDevice, st);
    if (err != cudaSuccess) return kvattn::cuda_fail(err);
  }
  return KVATTN_OK;
}
