// mla_decode_kernel<48, 3, *>: 48 query rows per MMA N-tile, 3-stage ring of 96-position
// tiles; the plain decode and the shared-prefix cascade.
#include "mla_decode_instantiate.cuh"

namespace pmla {
int launch_decode_ng48(const CUtensorMap& q_lat, const CUtensorMap& q_rope,
                       const DecodeParams& prm, int grid, cudaStream_t stream) {
  return launch_decode_impl<48, 3, kSchedCascade>(q_lat, q_rope, prm, grid, stream);
}
}  // namespace pmla
