// mla_selftest_bounded_wait: runs the pipeline's bounded mbarrier wait (ptx.cuh mbar_wait,
// the wait every decode role uses) on a barrier that nothing ever arrives at, with a short
// limit, so that a test can see on the GPU what a wait that runs out does: it returns
// false, raises the CTA's abort flag and sets the timeout bit of the error word, and the
// kernel then returns normally.  No fault, trap or hang is involved: the barrier is a
// valid, initialised one in shared memory, and the wait ends by its clock limit.
#include <cuda_runtime.h>

#include "../../include/paged_mla.h"
#include "ptx.cuh"

namespace {

__global__ void wait_selftest_kernel(int* err_word, int* result, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  const uint32_t b = pmla::smem_u32(&bar);
  pmla::mbar_init(b, 1);   // one arrival completes phase 0; none ever comes
  abort_flag = 0;
  pmla::fence_mbar_init();
  const unsigned long long t0 = pmla::globaltimer_ns();
  const bool ok = pmla::mbar_wait(b, 0, &abort_flag, err_word, limit_ns);
  const unsigned long long t1 = pmla::globaltimer_ns();
  result[0] = ok ? 1 : 0;
  result[1] = abort_flag;
  result[2] = static_cast<int>((t1 - t0) / 1000ull);   // microseconds spent in the wait
}

}  // namespace

extern "C" int mla_selftest_bounded_wait(int32_t* error_word, int32_t* result, int64_t limit_ns,
                                         mla_stream_t stream_) {
  if (!error_word || !result || limit_ns < 1000 || limit_ns > 100000000) return MLA_ERR_INVALID_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  wait_selftest_kernel<<<1, 32, 0, stream>>>(error_word, result,
                                            static_cast<unsigned long long>(limit_ns));
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
