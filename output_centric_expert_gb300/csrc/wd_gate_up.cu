// moe_gate_up: the launch of the first kernel of the layer -- the choice of
// slots per warp, the kernels that read H at run time, and the dispatch to
// the kernels compiled for fixed H (wd_gate_up_fixed.cu).
#include "wd_gate_up.cuh"

namespace wd {
namespace {

// Slots per warp of moe_gate_up for small batches: the fewest that make the
// grid a single wave at 3 CTAs per SM, as long as a warp has at most 8 (slot,
// segment) units to stream one after the other (measured: Q30 B=2 19.5 ->
// 18.1 us, B=4 29.7 -> 28.3, Q235 B=1 34.6 -> 33.0; 32 units per warp for the
// DeepSeek-V3-shaped layer at B=1 was slower); 0 if there is none.
int small_batch_spw(int B, int top_k, int I, int nseg) {
  const int sms = sm_count();
  const int small[4] = {1, 2, 4, 8};
  for (int v : small) {
    if ((v > top_k && v > 1) || v * nseg > 8) break;
    const int64_t ctas = (int64_t)B * ((top_k + v - 1) / v) * (I / kWarpsPerCta);
    if (ctas <= 3 * sms) return v;
  }
  return 0;
}

// Otherwise: as many as keep at least kMinCtasPerSm CTAs per SM.
int pick_spw(int B, int top_k, int I) {
  const int sms = sm_count();
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
  int spw = small_batch_spw(B, s->top_k, s->I, nseg), ctas_per_sm = 3;
  if (spw == 0) {
    spw = pick_spw(B, s->top_k, s->I);
    // Up to 1.5 E pairs for H = 2048 (where 8 slots at three CTAs win from 28
    // tokens) and below 1.625 E pairs from H = 4096 (the batches the layer runs
    // this kernel on, and moe_gate_up's own calls a little beyond), for the
    // rows compiled with fixed length: four CTAs
    // per SM (64 registers) with 4 (slot, segment) units per warp (H = 2048;
    // H = 4096 up to E pairs or with top_k < 4) or 8 (H = 4096 beyond E
    // pairs; H = 7168). Measured on GB300 in the layer (CUDA graph, against
    // the slots per warp the CTA-count rule gives at three CTAs per SM):
    // Qwen-3-30B-A3B shape B=8..24 3-6 % faster (B=16 75.1 -> 70.9 us),
    // slower from 28 tokens; Qwen-3-235B-A22B shape B=4..20 3-8 % faster
    // (B=12 239.0 -> 221.1 us); DeepSeek-V3 shape B=4..40 2-12 % faster (B=32
    // 1347.7 -> 1188.7 us); Mixtral shape (top-2) B=2..5 2-5 % faster. Each
    // intermediate is the same bit for bit.
    const int64_t P = (int64_t)B * s->top_k, E = s->E;
    if (s->H == 2048 ? 2 * P <= 3 * E : 8 * P < 13 * E) {
      if (s->H == 2048 && s->top_k >= 4) {
        spw = 4;
        ctas_per_sm = 4;
      } else if (s->H == 4096 && s->top_k >= 2) {
        spw = (P <= E || s->top_k < 4) ? 2 : 4;
        ctas_per_sm = 4;
      } else if (s->H == 7168 && s->top_k >= 2) {
        spw = 2;
        ctas_per_sm = 4;
      }
    }
  }
  if (launch_gate_up_fixed_h(s, w, x, ids, B, h, err, st, route, spw, ctas_per_sm, &rc))
    return rc;
  if (nseg == 1) rc = launch_gate_up_spw<1>(s, w, x, ids, B, h, err, st, route, spw);
  else if (nseg == 2) rc = launch_gate_up_spw<2>(s, w, x, ids, B, h, err, st, route, spw);
  else rc = launch_gate_up_spw<4>(s, w, x, ids, B, h, err, st, route, spw);
  return rc;
}

}  // namespace wd
