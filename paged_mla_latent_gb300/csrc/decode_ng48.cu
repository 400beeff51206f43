// mla_decode_kernel<48, *, *>: 48 query rows per MMA N-tile.  The plain decode streams its
// rows from HBM and runs a 3-stage ring of 96-position tiles (more bytes in flight); the
// shared-prefix cascade, whose prefix rows mostly come from L2 and whose time goes to the
// 48-column softmax, keeps 2 stages of 128 positions (fewer tiles per position).
#include "mla_decode_instantiate.cuh"

namespace pmla {
int launch_decode_ng48(const CUtensorMap& q_lat, const CUtensorMap& q_rope,
                       const DecodeParams& prm, int grid, cudaStream_t stream) {
  if (prm.sp.mode == kSchedCascade)
    return launch_decode_mode<48, 2, kSchedCascade>(q_lat, q_rope, prm, grid, stream);
  return launch_decode_impl<48, 3, kSchedWhole>(q_lat, q_rope, prm, grid, stream);
}
}  // namespace pmla
