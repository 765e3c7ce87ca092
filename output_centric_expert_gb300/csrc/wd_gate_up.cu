// moe_gate_up: the launch of the first kernel of the layer -- the choice of
// slots per warp, the kernels that read H at run time, and the dispatch to
// the kernels compiled for fixed H (wd_gate_up_fixed.cu).
#include "wd_gate_up.cuh"

namespace wd {
namespace {

// Slots per warp of moe_gate_up. Small batches: the fewest that make the grid
// a single wave at 3 CTAs per SM, as long as a warp has at most 8 (slot,
// segment) units to stream one after the other (measured: Q30 B=2 19.5 ->
// 18.1 us, B=4 29.7 -> 28.3, Q235 B=1 34.6 -> 33.0; 32 units per warp for the
// DeepSeek-V3-shaped layer at B=1 was slower). Otherwise as many as keep at
// least kMinCtasPerSm CTAs per SM.
int pick_spw(int B, int top_k, int I, int nseg) {
  const int sms = sm_count();
  const int small[4] = {1, 2, 4, 8};
  for (int v : small) {
    if ((v > top_k && v > 1) || v * nseg > 8) break;
    const int64_t ctas = (int64_t)B * ((top_k + v - 1) / v) * (I / kWarpsPerCta);
    if (ctas <= 3 * sms) return v;
  }
  const int spws[4] = {8, 4, 2, 1};
  for (int v : spws) {
    if (v > top_k) continue;
    const int64_t ctas = (int64_t)B * ((top_k + v - 1) / v) * (I / kWarpsPerCta);
    if (ctas >= (int64_t)kMinCtasPerSm * sms) return v;
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
  const int nseg = ((s->H >> 5) + kSegBlocks - 1) / kSegBlocks;  // 2048-element row segments
  const int spw = pick_spw(B, s->top_k, s->I, nseg);
  if (launch_gate_up_fixed_h(s, w, x, ids, B, h, err, st, route, spw, &rc)) return rc;
  if (nseg == 1) rc = launch_gate_up_spw<1>(s, w, x, ids, B, h, err, st, route, spw);
  else if (nseg == 2) rc = launch_gate_up_spw<2>(s, w, x, ids, B, h, err, st, route, spw);
  else rc = launch_gate_up_spw<4>(s, w, x, ids, B, h, err, st, route, spw);
  return rc;
}

}  // namespace wd
