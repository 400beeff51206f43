// Host launchers of the decode kernel instantiations (one translation unit each).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "mla_decode_kernel.cuh"

namespace pmla {

// Launch mla_decode_kernel<NG, stages> on `grid` CTAs; sets the kernel's dynamic shared
// memory limit on first use per device.  Returns 0 or an mla_status_t.
int launch_decode_ng16(const CUtensorMap& q_lat, const CUtensorMap& q_rope,
                       const DecodeParams& prm, int grid, cudaStream_t stream);
int launch_decode_ng32(const CUtensorMap& q_lat, const CUtensorMap& q_rope,
                       const DecodeParams& prm, int grid, cudaStream_t stream);
int launch_decode_ng48(const CUtensorMap& q_lat, const CUtensorMap& q_rope,
                       const DecodeParams& prm, int grid, cudaStream_t stream);
// mla_decode_rows96_kernel (mla_decode_rows96.cuh): 96 rows, any schedule mode.
int launch_decode_ng96(const CUtensorMap& q_lat, const CUtensorMap& q_rope,
                       const DecodeParams& prm, int grid, cudaStream_t stream);

}  // namespace pmla
