// moe_gate_up: the launch of the first kernel of the layer -- the choice of
// slots per warp, the kernels that read H at run time, and the dispatch to
// the kernels compiled for fixed H (wd_gate_up_fixed.cu).
#include "wd_gate_up.cuh"

namespace wd {
namespace {

// Slots per warp of moe_gate_up: as many as keep at least kMinCtas CTAs.
int pick_spw(int B, int top_k, int I) {
  const int spws[4] = {8, 4, 2, 1};
  for (int v : spws) {
    if (v > top_k) continue;
    const int64_t ctas = (int64_t)B * ((top_k + v - 1) / v) * (I / kWarpsPerCta);
    if (ctas >= kMinCtas) return v;
  }
  return 1;
}

// The kernels that read H at run time (the fixed-H ones are in
// wd_gate_up_fixed.cu).
template <int SPW, int NSEG>
moe_status launch_gate_up_full(const moe_shape* s, const moe_weights* w, const uint16_t* x,
                               const int32_t* ids, int32_t B, uint16_t* h, int32_t* err,
                               cudaStream_t st, RouteArgs route) {
  if ((s->H >> 5) % kSegBlocks == 0)
    return launch_gate_up<SPW, NSEG, true, 0>(s, w, x, ids, B, h, err, st, route);
  return launch_gate_up<SPW, NSEG, false, 0>(s, w, x, ids, B, h, err, st, route);
}

template <int NSEG>
moe_status launch_gate_up_spw(const moe_shape* s, const moe_weights* w, const uint16_t* x,
                              const int32_t* ids, int32_t B, uint16_t* h, int32_t* err,
                              cudaStream_t st, RouteArgs route, int spw) {
  switch (spw) {
    case 8: return launch_gate_up_full<8, NSEG>(s, w, x, ids, B, h, err, st, route);
    case 4: return launch_gate_up_full<4, NSEG>(s, w, x, ids, B, h, err, st, route);
    case 2: return launch_gate_up_full<2, NSEG>(s, w, x, ids, B, h, err, st, route);
    default: return launch_gate_up_full<1, NSEG>(s, w, x, ids, B, h, err, st, route);
  }
}

}  // namespace

moe_status launch_gate_up_kernels(const moe_shape* s, const moe_weights* w, const uint16_t* x,
                                  const int32_t* ids, int32_t B, uint16_t* h, int32_t* err,
                                  cudaStream_t st, RouteArgs route) {
  moe_status rc;
  const int spw = pick_spw(B, s->top_k, s->I);
  if (launch_gate_up_fixed_h(s, w, x, ids, B, h, err, st, route, spw, &rc)) return rc;
  const int nseg = ((s->H >> 5) + kSegBlocks - 1) / kSegBlocks;  // 2048-element row segments
  if (nseg == 1) rc = launch_gate_up_spw<1>(s, w, x, ids, B, h, err, st, route, spw);
  else if (nseg == 2) rc = launch_gate_up_spw<2>(s, w, x, ids, B, h, err, st, route, spw);
  else rc = launch_gate_up_spw<4>(s, w, x, ids, B, h, err, st, route, spw);
  return rc;
}

}  // namespace wd
