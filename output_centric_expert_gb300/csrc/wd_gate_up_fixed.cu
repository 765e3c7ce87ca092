// moe_gate_up kernels compiled for fixed row lengths H: the hidden sizes of
// the Qwen3-30B-A3B-, Qwen3-235B-A22B- (and Mixtral-) and DeepSeek-V3-shaped
// layers. With H a constant the row strides and activation offsets are
// immediates of the loads (about 5 % fewer instructions per weight).
#include "wd_gate_up.cuh"

namespace wd {
namespace {

template <int SPW>
bool launch_fixed(const moe_shape* s, const moe_weights* w, const uint16_t* x, const int32_t* ids,
                  int32_t B, uint16_t* h, int32_t* err, cudaStream_t st, RouteArgs route,
                  moe_status* rc) {
  switch (s->H) {
    case 2048: *rc = launch_gate_up<SPW, 1, true, 2048>(s, w, x, ids, B, h, err, st, route); return true;
    case 4096: *rc = launch_gate_up<SPW, 2, true, 4096>(s, w, x, ids, B, h, err, st, route); return true;
    case 7168: *rc = launch_gate_up<SPW, 4, false, 7168>(s, w, x, ids, B, h, err, st, route); return true;
    default: return false;
  }
}

// The same at four CTAs per SM (64 registers), for up to 4 slots per warp.
template <int SPW>
bool launch_fixed4(const moe_shape* s, const moe_weights* w, const uint16_t* x, const int32_t* ids,
                   int32_t B, uint16_t* h, int32_t* err, cudaStream_t st, RouteArgs route,
                   moe_status* rc) {
  switch (s->H) {
    case 2048: *rc = launch_gate_up<SPW, 1, true, 2048, 4>(s, w, x, ids, B, h, err, st, route); return true;
    case 4096: *rc = launch_gate_up<SPW, 2, true, 4096, 4>(s, w, x, ids, B, h, err, st, route); return true;
    case 7168: *rc = launch_gate_up<SPW, 4, false, 7168, 4>(s, w, x, ids, B, h, err, st, route); return true;
    default: return false;
  }
}

}  // namespace

bool launch_gate_up_fixed_h(const moe_shape* s, const moe_weights* w, const uint16_t* x,
                            const int32_t* ids, int32_t B, uint16_t* h, int32_t* err,
                            cudaStream_t st, RouteArgs route, int spw, int ctas_per_sm,
                            moe_status* rc) {
  if (ctas_per_sm == 4) {
    if (spw == 4) return launch_fixed4<4>(s, w, x, ids, B, h, err, st, route, rc);
    if (spw == 2) return launch_fixed4<2>(s, w, x, ids, B, h, err, st, route, rc);
  }
  switch (spw) {
    case 8: return launch_fixed<8>(s, w, x, ids, B, h, err, st, route, rc);
    case 4: return launch_fixed<4>(s, w, x, ids, B, h, err, st, route, rc);
    case 2: return launch_fixed<2>(s, w, x, ids, B, h, err, st, route, rc);
    default: return launch_fixed<1>(s, w, x, ids, B, h, err, st, route, rc);
  }
}

}  // namespace wd
