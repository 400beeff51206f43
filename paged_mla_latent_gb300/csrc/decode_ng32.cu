// mla_decode_kernel<32, 3, kSchedWhole>: 32 query rows per MMA N-tile, 3-stage ring of
// 96-position tiles.
#include "mla_decode_instantiate.cuh"

namespace pmla {
int launch_decode_ng32(const CUtensorMap& q_lat, const CUtensorMap& q_rope,
                       const DecodeParams& prm, int grid, cudaStream_t stream) {
  return launch_decode_impl<32, 3, kSchedWhole>(q_lat, q_rope, prm, grid, stream);
}
}  // namespace pmla
