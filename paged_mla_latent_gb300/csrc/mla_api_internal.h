// Library-internal host entry points shared between translation units (not part of the
// C ABI).
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "../../include/paged_mla.h"

namespace pmla {

// cuTensorMapEncodeTiled, found once through the runtime's driver entry point (no libcuda
// link), or null if the driver does not provide it.
void* tensor_map_encoder();

// Every host-side check mla_decode makes on these arguments (shapes, dtypes, strides,
// scalars, workspace size and alignment), without enqueuing anything.  Returns MLA_OK or
// the status mla_decode would return before its first launch.
int check_decode_call(const mla_tensor_t* q, const mla_tensor_t* kv_buffer, const mla_tensor_t* o,
                      const mla_tensor_t* qo_indptr, const mla_tensor_t* kv_indptr,
                      const mla_tensor_t* kv_indices, const mla_tensor_t* kv_last_page_lens,
                      int32_t max_seqlen_q, float sm_scale, const mla_tensor_t* q_scale,
                      const mla_tensor_t* kv_scale, int32_t num_kv_splits,
                      const mla_tensor_t* lse_out, void* workspace, size_t workspace_bytes);

}  // namespace pmla
