// mla_expand_shared_prefix_indices: the full page table of a shared-prefix batch, built on
// the device from the compact form a prefix cache holds.
//
// "[Kimi-K3 MLA TP8] MLA performance" §1 "Environment" describes decode batches whose
// requests share a long prefix of cache entries (the prefix cache), and §5.4 raises reusing
// it across requests.  A caller that knows the shared pages keeps them once and each
// request's own pages after them; mla_decode_shared_prefix reads the CSR page table of §4.1
// (kv_indptr, kv_indices), in which every request lists the shared pages again.  Handing the
// compact form to the device and expanding it there moves the shared ids over the host link
// once instead of once per request (for the concurrency-16 step: 0.5 MB of ids instead of
// 4.4 MB).
//
// Index plumbing, memory-bound: block (x, b) copies, grid-stride over x, request b's ids;
// consecutive threads write consecutive entries.  Request b's entries start at
// b * n_shared + (own_indptr[b] - own_indptr[0]), computed without a scan over the batch.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/paged_mla.h"

namespace {

constexpr int kThreads = 256;
constexpr int kBlocksPerRequest = 16;
constexpr int kErrBadIndptr = 2;    // the library's device error bits (ptx.cuh)
constexpr int kErrBadOutput = 8;

__global__ void __launch_bounds__(kThreads)
    expand_prefix_kernel(const int32_t* __restrict__ shared, int64_t n_shared,
                         const int32_t* __restrict__ own_indptr,
                         const int32_t* __restrict__ own, int64_t own_len, int B,
                         int32_t* __restrict__ kv_indptr, int32_t* __restrict__ kv_indices,
                         int64_t kv_cap, int* err) {
  const int b = blockIdx.y;
  const int64_t o0 = own_indptr[0];
  const int64_t ob = own_indptr[b];
  const int64_t oe = own_indptr[b + 1];
  if (o0 < 0 || ob < o0 || oe < ob || oe > own_len) {   // own_indptr: offsets into own
    if (blockIdx.x == 0 && threadIdx.x == 0 && err) atomicOr(err, kErrBadIndptr);
    return;
  }
  const int64_t base = static_cast<int64_t>(b) * n_shared + (ob - o0);
  const int64_t len = n_shared + (oe - ob);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    const int64_t end = base + len;
    if (end > INT32_MAX || end > kv_cap) {
      if (err) atomicOr(err, kErrBadOutput);
    }
    if (end <= INT32_MAX) {
      kv_indptr[b] = static_cast<int32_t>(base);
      if (b == B - 1) kv_indptr[B] = static_cast<int32_t>(end);
    }
  }
  const int64_t step = static_cast<int64_t>(gridDim.x) * kThreads;
  for (int64_t j = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; j < len; j += step) {
    const int32_t v = j < n_shared ? shared[j] : own[ob + (j - n_shared)];
    const int64_t at = base + j;
    if (at < kv_cap) {
      kv_indices[at] = v;
    } else if (err) {
      atomicOr(err, kErrBadOutput);
      break;
    }
  }
}

bool is_i32_vec(const mla_tensor_t* t, int64_t* len) {
  if (!t || !t->ptr || t->dtype != MLA_DTYPE_INT32 || t->ndim != 1) return false;
  if (t->shape[0] < 0 || (t->shape[0] > 1 && t->stride[0] != 1)) return false;
  if (reinterpret_cast<uintptr_t>(t->ptr) % 4 != 0) return false;
  *len = t->shape[0];
  return true;
}

}  // namespace

extern "C" int mla_expand_shared_prefix_indices(const mla_tensor_t* shared_indices,
                                                const mla_tensor_t* own_indptr,
                                                const mla_tensor_t* own_indices,
                                                const mla_tensor_t* kv_indptr,
                                                const mla_tensor_t* kv_indices,
                                                int32_t* error_word, mla_stream_t stream_) {
  int64_t n_shared = 0, n_ip = 0, n_own = 0, n_kvp = 0, n_kv = 0;
  if (!is_i32_vec(own_indptr, &n_ip) || n_ip < 1) return MLA_ERR_INVALID_ARG;
  if (!is_i32_vec(kv_indptr, &n_kvp) || n_kvp != n_ip) return MLA_ERR_INVALID_ARG;
  if (!is_i32_vec(kv_indices, &n_kv)) return MLA_ERR_INVALID_ARG;
  if (!is_i32_vec(own_indices, &n_own)) {
    // an empty own list may come as a null pointer
    if (!own_indices || own_indices->ndim != 1 || own_indices->shape[0] != 0 ||
        own_indices->dtype != MLA_DTYPE_INT32)
      return MLA_ERR_INVALID_ARG;
    n_own = 0;
  }
  if (!is_i32_vec(shared_indices, &n_shared)) {
    if (!shared_indices || shared_indices->ndim != 1 || shared_indices->shape[0] != 0 ||
        shared_indices->dtype != MLA_DTYPE_INT32)
      return MLA_ERR_INVALID_ARG;
    n_shared = 0;
  }
  const int64_t B = n_ip - 1;
  if (B == 0) return MLA_OK;
  if (B > 65535) return MLA_ERR_UNSUPPORTED;   // one grid row per request
  if (B * n_shared > n_kv) return MLA_ERR_INVALID_ARG;   // cannot hold even the shared ids
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const dim3 grid(kBlocksPerRequest, static_cast<unsigned>(B));
  expand_prefix_kernel<<<grid, kThreads, 0, stream>>>(
      static_cast<const int32_t*>(shared_indices->ptr), n_shared,
      static_cast<const int32_t*>(own_indptr->ptr),
      static_cast<const int32_t*>(n_own > 0 ? own_indices->ptr : nullptr), n_own,
      static_cast<int>(B), static_cast<int32_t*>(kv_indptr->ptr),
      static_cast<int32_t*>(kv_indices->ptr), n_kv, error_word);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
