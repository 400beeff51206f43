// mla_decode_kernel<32, 2, kSchedWhole>: 32 query rows per MMA N-tile, 2-stage cache ring.
#include "mla_decode_instantiate.cuh"

namespace pmla {
int launch_decode_ng32(const CUtensorMap& q_lat, const CUtensorMap& q_rope,
                       const DecodeParams& prm, int grid, cudaStream_t stream) {
  return launch_decode_impl<32, 2, kSchedWhole>(q_lat, q_rope, prm, grid, stream);
}
}  // namespace pmla
