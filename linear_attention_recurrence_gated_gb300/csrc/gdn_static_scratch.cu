// gdn_fwd_static_scratch: the forward pass for callers that cannot allocate
// device memory.  The status record that gdn_fwd keeps in the caller's
// workspace lives here in a file-scope __device__ array instead, so the
// caller passes only inputs and outputs.  No cudaMalloc/cudaFree is called.
#include <mutex>
#include <string.h>

#include "gdn_internal.cuh"

namespace {

// Scratch for one call: the device status record.  Every GPU that loads the
// library holds these bytes until the process exits; all calls on a device
// share them.
constexpr size_t kStaticScratchBytes = 256;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the array on the current device.  Host code may not use
// the symbol itself as a device pointer, so the address comes from
// cudaGetSymbolAddress with the device current.  Outside stream capture it is
// looked up again on every call (the lookup allocates nothing), so a context
// that was reset and created anew is seen; during capture the address cached
// by the last uncaptured call on this device is used, since the lookup could
// initialise state that capture does not allow.
gdn_status scratch_address(cudaStream_t s, void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return GDN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return GDN_ERR_UNSUPPORTED;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) return GDN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (cap == cudaStreamCaptureStatusNone || g_scratch_addr[dev] == nullptr) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || ptr == nullptr)
      return GDN_ERR_CUDA;
    g_scratch_addr[dev] = ptr;
  }
  *out = g_scratch_addr[dev];
  return GDN_OK;
}

}  // namespace

extern "C" gdn_status gdn_fwd_static_scratch(
    const void *q, const void *k, const void *v, const float *g, const void *beta,
    const float *initial_state, const int32_t *cu_seqlens, void *o, float *final_state,
    const float *D_skip, const float *out_gate, int32_t batch, int32_t seq_len,
    int32_t num_heads, int32_t head_dim_k, int32_t head_dim_v, int32_t num_seqs, int32_t chunk_size, gdn_dtype dtype, uint32_t flags, int32_t check,
    void *stream) {
  const size_t need =
      gdn_fwd_workspace_size(num_seqs, num_heads, head_dim_k, head_dim_v, flags);
  if (need == 0) return GDN_ERR_INVALID_ARG;
  if (need > kStaticScratchBytes) return GDN_ERR_WORKSPACE;  // beyond the static maximum

  cudaStream_t s = (cudaStream_t)stream;
  void *scratch = nullptr;
  gdn_status st = scratch_address(s, &scratch);
  if (st != GDN_OK) return st;

  // every host-side check of gdn_fwd runs before anything is enqueued
  gdn::FwdCall call;
  st = gdn::fwd_validate(q, k, v, g, beta, initial_state, cu_seqlens, o, final_state, D_skip,
                         out_gate, batch, seq_len, num_heads, head_dim_k, head_dim_v, num_seqs,
                         chunk_size, dtype, flags, scratch, kStaticScratchBytes, &call);
  if (st != GDN_OK) return st;

  // The array keeps the previous call's contents: the status must start at zero.
  if (cudaMemsetAsync(scratch, 0, kStaticScratchBytes, s) != cudaSuccess) return GDN_ERR_CUDA;
  st = gdn::fwd_launch(call, s);
  if (st != GDN_OK || !check) return st;

  gdn::DeviceStatus rec;
  memset(&rec, 0, sizeof rec);
  if (cudaMemcpyAsync(&rec, scratch, sizeof rec, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return GDN_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return GDN_ERR_CUDA;
  if (rec.code == 0) return GDN_OK;
  return rec.code <= GDN_ERR_DEVICE_CHECK ? (gdn_status)rec.code : GDN_ERR_DEVICE_CHECK;
}
