// Host interface of the expert-grouped moe_gate_up kernel
// (wd_gate_up_grouped.cu), used by the C-ABI entry points in warp_decode.cu.
#pragma once

#include <cuda_runtime.h>

#include "warp_decode.h"

namespace wd {

// Whether the grouped kernel handles the shape, batch and weights:
// H % 256 == 0, I % 64 == 0, E <= 256, gu_scales 8-byte aligned (not checked
// when w is NULL), and its shared memory for B tokens within the limit.
bool gate_up_grouped_supported(const moe_shape* s, const moe_weights* w, int32_t B);

// Launch it on `st` (expert ids only, no routing from logits); the arguments
// have been validated by the entry point. dependent: launch as a programmatic
// dependent of the preceding kernel (the router that writes the ids; the
// kernel waits for it before reading them). Returns MOE_OK or an error status.
moe_status launch_gate_up_grouped(const moe_shape* s, const moe_weights* w, const uint16_t* x,
                                  const int32_t* ids, int32_t B, uint16_t* h, int32_t* err,
                                  cudaStream_t st, bool dependent = false);

}  // namespace wd
