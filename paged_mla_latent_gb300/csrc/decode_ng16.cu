// mla_decode_kernel<16, 3, kSchedWhole>: 16 query rows per MMA N-tile, 3-stage cache ring.
#include "mla_decode_instantiate.cuh"

namespace pmla {
int launch_decode_ng16(const CUtensorMap& q_lat, const CUtensorMap& q_rope,
                       const DecodeParams& prm, int grid, cudaStream_t stream) {
  return launch_decode_impl<16, 3, kSchedWhole>(q_lat, q_rope, prm, grid, stream);
}
}  // namespace pmla
