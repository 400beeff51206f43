// mla_decode_rows96_kernel<*>: 96 query rows per pass over the cache (query rows on the
// tensor-memory lanes, block-scaled PV), 4-stage ring of 64-position tiles; the plain decode
// and the shared-prefix cascade.
#include <mutex>

#include "../../include/paged_mla.h"
#include "mla_decode_launch.h"
#include "mla_decode_rows96.cuh"

namespace pmla {
namespace {

template <int MODE>
int launch_rows96(const CUtensorMap& q_lat, const CUtensorMap& q_rope, const DecodeParams& prm,
                  int grid, cudaStream_t stream) {
  using LY = Rows96Layout;
  static std::mutex mu;
  static bool attr_set[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MLA_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (!attr_set[dev]) {
      if (cudaFuncSetAttribute(mla_decode_rows96_kernel<MODE>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               LY::kSmemBytes) != cudaSuccess)
        return MLA_ERR_CUDA;
      attr_set[dev] = true;
    }
  }
  mla_decode_rows96_kernel<MODE><<<grid, LY::kThreads, LY::kSmemBytes, stream>>>(q_lat, q_rope, prm);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

}  // namespace

int launch_decode_ng96(const CUtensorMap& q_lat, const CUtensorMap& q_rope,
                       const DecodeParams& prm, int grid, cudaStream_t stream) {
  switch (prm.sp.mode) {
    case kSchedWhole: return launch_rows96<kSchedWhole>(q_lat, q_rope, prm, grid, stream);
    case kSchedCascade: return launch_rows96<kSchedCascade>(q_lat, q_rope, prm, grid, stream);
    case kSchedCascadePaged:
      return launch_rows96<kSchedCascadePaged>(q_lat, q_rope, prm, grid, stream);
    default: return MLA_ERR_UNSUPPORTED;
  }
}

}  // namespace pmla
