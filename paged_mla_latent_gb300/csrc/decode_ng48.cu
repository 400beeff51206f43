// mla_decode_kernel<48, 2, *>: 48 query rows per MMA N-tile, 2-stage cache ring; the plain
// decode and the shared-prefix cascade.
#include "mla_decode_instantiate.cuh"

namespace pmla {
int launch_decode_ng48(const CUtensorMap& q_lat, const CUtensorMap& q_rope,
                       const DecodeParams& prm, int grid, cudaStream_t stream) {
  return launch_decode_impl<48, 2, kSchedCascade>(q_lat, q_rope, prm, grid, stream);
}
}  // namespace pmla
