// Shared body of the per-instantiation launcher translation units.
#pragma once

#include <mutex>

#include "../../include/paged_mla.h"
#include "mla_decode_launch.h"

namespace pmla {

template <int NG, int STAGES, int MODE>
int launch_decode_mode(const CUtensorMap& q_lat, const CUtensorMap& q_rope,
                       const DecodeParams& prm, int grid, cudaStream_t stream) {
  using LY = DecodeLayout<NG, STAGES>;
  static std::mutex mu;
  static bool attr_set[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MLA_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (!attr_set[dev]) {
      if (cudaFuncSetAttribute(mla_decode_kernel<NG, STAGES, MODE>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               LY::kSmemBytes) != cudaSuccess)
        return MLA_ERR_CUDA;
      attr_set[dev] = true;
    }
  }
  mla_decode_kernel<NG, STAGES, MODE><<<grid, LY::kThreads, LY::kSmemBytes, stream>>>(
      q_lat, q_rope, prm);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

// The plain decode, or (CASCADE = kSchedCascade) also the shared-prefix cascade on pages of
// one token (kSchedCascade) and of several (kSchedCascadePaged).
template <int NG, int STAGES, int CASCADE>
int launch_decode_impl(const CUtensorMap& q_lat, const CUtensorMap& q_rope,
                       const DecodeParams& prm, int grid, cudaStream_t stream) {
  if (prm.sp.mode == kSchedWhole)
    return launch_decode_mode<NG, STAGES, kSchedWhole>(q_lat, q_rope, prm, grid, stream);
  if constexpr (CASCADE == kSchedCascade) {
    if (prm.sp.mode == kSchedCascade)
      return launch_decode_mode<NG, STAGES, kSchedCascade>(q_lat, q_rope, prm, grid, stream);
    if (prm.sp.mode == kSchedCascadePaged)
      return launch_decode_mode<NG, STAGES, kSchedCascadePaged>(q_lat, q_rope, prm, grid, stream);
  }
  return MLA_ERR_UNSUPPORTED;
}

}  // namespace pmla
