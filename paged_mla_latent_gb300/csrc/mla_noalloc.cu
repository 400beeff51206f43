// mla_decode_noalloc: the decode call for callers that must not allocate device memory.
//
// Some callers cannot call cudaMalloc (or cannot hand this library a scratch buffer):
// a plug-in running inside a serving engine whose device memory is owned by the engine's
// own pool, or a hook that only ever receives its input and output tensors.  For them
// the split-KV partials and the device error words live in one fixed, file-scope device
// array instead of a caller-provided workspace.  The array is part of this library's
// module, so every GPU that loads the library holds it (MLA_NOALLOC_SCRATCH_BYTES) until
// the process exits.  Nothing here allocates: the call looks up the array's device
// address (once per device), runs every host-side check of the decode, and only then
// clears the error words, runs the ordinary decode path on the array, and optionally
// copies the error word to the caller.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/paged_mla.h"
#include "mla_api_internal.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr size_t kErrorBytes = 256;   // device error words at the start of the scratch

// Split-KV partials + error words of mla_decode_noalloc.  Shared by every call on a device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MLA_NOALLOC_SCRATCH_BYTES];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices];   // device address of g_noalloc_scratch, per device

// Device address of the scratch array on the current device (looked up on first use).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MLA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    // The host-side name g_noalloc_scratch is only a stand-in; the kernels need the
    // address the runtime assigned on this device.
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return MLA_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MLA_OK;
}

}  // namespace

extern "C" int mla_decode_noalloc(const mla_tensor_t* q, const mla_tensor_t* kv_buffer,
                                  const mla_tensor_t* o, const mla_tensor_t* qo_indptr,
                                  const mla_tensor_t* kv_indptr, const mla_tensor_t* kv_indices,
                                  const mla_tensor_t* kv_last_page_lens, int32_t max_seqlen_q,
                                  float sm_scale, const mla_tensor_t* q_scale,
                                  const mla_tensor_t* kv_scale, int32_t num_kv_splits,
                                  const mla_tensor_t* lse_out, int32_t* error_out,
                                  mla_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (!q || !qo_indptr || q->ndim != 3 || qo_indptr->ndim != 1 || qo_indptr->shape[0] < 1)
    return MLA_ERR_INVALID_ARG;
  // Scratch this call needs, on the current device, against the fixed array.
  size_t need = 0;
  int rc = mla_get_workspace_size(static_cast<int32_t>(qo_indptr->shape[0] - 1),
                                  static_cast<int32_t>(q->shape[1]), max_seqlen_q, num_kv_splits,
                                  0, &need);
  if (rc != MLA_OK) return rc;
  if (need > static_cast<size_t>(MLA_NOALLOC_SCRATCH_BYTES)) return MLA_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  if ((rc = scratch_address(&scratch)) != MLA_OK) return rc;
  // Argument errors come back before anything is enqueued (the memset below included).
  rc = pmla::check_decode_call(q, kv_buffer, o, qo_indptr, kv_indptr, kv_indices,
                               kv_last_page_lens, max_seqlen_q, sm_scale, q_scale, kv_scale,
                               num_kv_splits, lse_out, scratch,
                               static_cast<size_t>(MLA_NOALLOC_SCRATCH_BYTES));
  if (rc != MLA_OK) return rc;
  // The error words must start at zero; the partials are always written before read.
  if (cudaMemsetAsync(scratch, 0, kErrorBytes, stream) != cudaSuccess) return MLA_ERR_CUDA;
  rc = mla_decode(q, kv_buffer, o, qo_indptr, kv_indptr, kv_indices, kv_last_page_lens,
                  max_seqlen_q, sm_scale, q_scale, kv_scale, num_kv_splits, lse_out, scratch,
                  static_cast<size_t>(MLA_NOALLOC_SCRATCH_BYTES), stream_);
  if (rc != MLA_OK) return rc;
  if (error_out != nullptr &&
      cudaMemcpyAsync(error_out, scratch, sizeof(int32_t), cudaMemcpyDeviceToDevice, stream) !=
          cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
}
