// Host interface of the expert-grouped moe_down kernel (wd_down_grouped.cu),
// used by the C-ABI entry points in warp_decode.cu.
#pragma once

#include <cuda_runtime.h>

#include "warp_decode.h"

namespace wd {

// Whether the grouped down kernel handles the shape, batch and weights:
// I % 256 == 0, E <= 256, 1 <= B <= 128, d_scales 8-byte aligned (not checked
// when w is NULL), and its shared memory within the per-CTA limit.
bool down_grouped_supported(const moe_shape* s, const moe_weights* w, int32_t B);

// Launch it on `st` (expert ids and routing weights given, no routing from
// logits); the arguments have been validated by the entry point. dependent:
// launched as a programmatic dependent of the gate/up kernel before it.
moe_status launch_down_grouped(const moe_shape* s, const moe_weights* w, const uint16_t* h,
                               const int32_t* ids, const float* wts, int32_t B, float* y,
                               int32_t* err, cudaStream_t st, bool dependent);

}  // namespace wd
