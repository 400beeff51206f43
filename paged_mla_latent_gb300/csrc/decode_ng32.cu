// mla_decode_kernel<32, 2, *>: 32 query rows per MMA N-tile, 2-stage cache ring; the plain
// decode and the shared-prefix cascade's suffix pass.
#include "mla_decode_instantiate.cuh"

namespace pmla {
int launch_decode_ng32(const CUtensorMap& q_lat, const CUtensorMap& q_rope,
                       const DecodeParams& prm, int grid, cudaStream_t stream) {
  return launch_decode_impl<32, 2, kSchedSuffix>(q_lat, q_rope, prm, grid, stream);
}
}  // namespace pmla
