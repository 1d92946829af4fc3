// decode_no_alloc.cu -- mla_decode for callers that cannot allocate device
// memory.  The scratch lives in one file-scope device array of fixed size
// (MLA_NO_ALLOC_WORKSPACE_BYTES); the caller passes only inputs and outputs.
#include <atomic>

#include "params.cuh"

// Shared by every call on a device and kept from call to call; each call
// rewrites everything it later reads (status word, plan, partials), so no
// clearing is needed between calls.
static __device__ __align__(256) unsigned char g_no_alloc_workspace[MLA_NO_ALLOC_WORKSPACE_BYTES];

namespace {
constexpr int kMaxDevices = 128;
// Device address of g_no_alloc_workspace, looked up once per device.
std::atomic<void*> g_workspace_addr[kMaxDevices];

void* workspace_address(int dev) {
  void* p = g_workspace_addr[dev].load(std::memory_order_acquire);
  if (p) return p;
  // In host code the array's name is only a host-side stand-in; the device
  // address must be asked for, with the device current.
  if (cudaGetSymbolAddress(&p, g_no_alloc_workspace) != cudaSuccess || !p) {
    cudaGetLastError();  // leave no sticky runtime error behind for the caller's next check
    return nullptr;
  }
  g_workspace_addr[dev].store(p, std::memory_order_release);
  return p;
}
}  // namespace

extern "C" int mla_decode_no_alloc(const mla_dims* d, const void* q_nope, const void* q_pe, const void* cache,
                                   const float* cache_scale_zero, int32_t num_pages, const int32_t* block_table,
                                   int32_t max_pages_per_seq, const int32_t* seq_lens, int32_t batch,
                                   const void* W_UK, const void* W_UV, float softmax_scale, int32_t num_splits,
                                   void* out, float* lse_out, int32_t* device_status, mla_stream_t stream) {
  const size_t need = mla_decode_workspace_size(d, batch, num_splits);
  if (need == 0) {  // the status mla_decode gives for the same arguments
    const int st = mla_check_dims(d);
    if (st != MLA_OK) return st;
    if (batch <= 0 || num_splits < 0 || (long long)batch * d->num_heads > MLA_MAX_QUERY_ROWS)
      return MLA_ERR_INVALID_ARG;
    return MLA_ERR_CUDA;  // valid arguments: the split count could not be resolved on this device
  }
  if (need > MLA_NO_ALLOC_WORKSPACE_BYTES) return MLA_ERR_WORKSPACE;  // larger than the fixed scratch
  if (device_status && (reinterpret_cast<uintptr_t>(device_status) & 3)) return MLA_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MLA_ERR_CUDA;
  void* ws = workspace_address(dev);
  if (!ws) return MLA_ERR_CUDA;
  const int st = mla_decode(d, q_nope, q_pe, cache, cache_scale_zero, num_pages, block_table, max_pages_per_seq,
                            seq_lens, batch, W_UK, W_UV, softmax_scale, num_splits, ws,
                            MLA_NO_ALLOC_WORKSPACE_BYTES, out, lse_out, stream);
  if (st != MLA_OK || !device_status) return st;
  // the status word sits at the start of the scratch; copy it out on the stream
  if (cudaMemcpyAsync(device_status, ws, sizeof(int32_t), cudaMemcpyDeviceToDevice,
                      reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
}
