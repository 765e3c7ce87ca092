// moe_gate_up kernel template and its launch, shared by wd_gate_up.cu (the
// kernels that read H at run time, and the dispatch) and wd_gate_up_fixed.cu
// (the kernels compiled for fixed H), which build in parallel.
#pragma once

#include "wd_device.cuh"

namespace wd {
namespace {

// ------------------------------------------------------------ moe_gate_up --
// grid.x = B * ceil(top_k / SPW) (token, slot group), grid.y = I / 8 (neuron
// block); 8 warps, warp w computes neuron n = 8*blockIdx.y + w for the SPW
// routed slots of its group. Dynamic shared memory: H f16 (the scaled x row).
//
// A warp's work is SPW * NSEG units (slot, segment of 2048 row elements),
// unrolled at compile time: load the unit's gate and up codes, then consume
// them. Each lane keeps one (gate, up) partial pair per slot; all of them are
// reduced together at the end and the SwiGLU epilogue of the SPW neurons runs
// once, in SPW lanes side by side.

struct GateUpUnit {
  Codes32 g[kSegBlocksPerLane], u[kSegBlocksPerLane];
  uint32_t sg[kSegBlocksPerLane], su[kSegBlocksPerLane];
};

// FULL: every segment is whole (H a multiple of 2048), so no block index
// needs checking against the row length.
// KH: the row length H fixed at compile time (0: taken from the argument). With
// it the row strides and the activation offsets are constants, which the
// loads take as immediates -- about 5 % fewer instructions per weight.
// MINB: CTAs per SM the registers are sized for (3: up to 85 per thread; 4:
// 64, for up to 4 slots per warp).
template <int SPW, int NSEG, bool FULL, int KH, int MINB = 3>
__global__ void __launch_bounds__(kThreads, MINB)
    moe_gate_up_kernel(const uint8_t* __restrict__ gu_codes,
                       const uint8_t* __restrict__ gu_scales,
                       const uint16_t* __restrict__ x, const int32_t* __restrict__ ids,
                       uint16_t* __restrict__ h, int32_t* __restrict__ err, int H_arg, int I,
                       int E, int top_k, RouteArgs route) {
  const int H = KH ? KH : H_arg;
  extern __shared__ uint4 xs[];
  __shared__ float red[kWarpsPerCta];
  const int lane = threadIdx.x & 31;
  const int groups = (top_k + SPW - 1) / SPW;
  const int t = blockIdx.x / groups;
  const int j0 = (blockIdx.x - t * groups) * SPW;
  const int n = blockIdx.y * kWarpsPerCta + (threadIdx.x >> 5);
  const int nblk = H >> 5;
  const int nslots = min(SPW, top_k - j0);

  // lane s < nslots holds the expert id of slot s; -1 marks "no slot".
  // moe_down is launched as a dependent of this kernel and reads the ids
  // before its own wait, so the dependents are released only once the ids
  // are complete (after the wait for a router that writes them; at once
  // otherwise).
  int e_lane;
  if (route.logits) {  // route the token here, from its logits (every warp routes: a
                       // barrier here, to route once per CTA, slowed the kernel for
                       // the 235B-shaped layer even when no logits are given)
    launch_dependents();
    int rid;
    float rw;
    warp_route(route.logits + (size_t)t * E, E, top_k, rid, rw);
    e_lane = __shfl_sync(0xFFFFFFFFu, rid, lane < nslots ? j0 + lane : 0);
    if (lane >= nslots) e_lane = -1;
  } else {
    wait_prerequisite();  // the ids are complete from here on (a router may write them)
    launch_dependents();
    e_lane = (lane < nslots) ? __ldg(ids + (size_t)t * top_k + j0 + lane) : -1;
  }

  auto load_unit = [&](int s, int seg, GateUpUnit& U) {
    const int e = __shfl_sync(0xFFFFFFFFu, e_lane, s);
    if (s >= nslots || e < 0 || e >= E) return;
    const size_t row = (size_t)e * I + n;
    const uint8_t* gc = gu_codes + row * 2 * (size_t)H;
    const uint8_t* sc = gu_scales + row * 2 * (size_t)nblk;
#pragma unroll
    for (int q = 0; q < kSegBlocksPerLane; ++q) {
      const int b = seg * kSegBlocks + q * 32 + lane;
      if (FULL || b < nblk) {
        U.g[q] = ld_codes32(gc + (size_t)b * 32);
        U.u[q] = ld_codes32(gc + H + (size_t)b * 32);
        U.sg[q] = __ldg(sc + b);
        U.su[q] = __ldg(sc + nblk + b);
      }
    }
  };

  float acc[2 * SPW];  // acc[s] gate, acc[SPW + s] up partials of slot s
#pragma unroll
  for (int i = 0; i < 2 * SPW; ++i) acc[i] = 0.0f;

  auto compute_unit = [&](int s, int seg, const GateUpUnit& U) {
    const int e = __shfl_sync(0xFFFFFFFFu, e_lane, s);
    if (s >= nslots || e < 0 || e >= E) return;
#pragma unroll
    for (int q = 0; q < kSegBlocksPerLane; ++q) {
      const int b = seg * kSegBlocks + q * 32 + lane;
      if (FULL || b < nblk) {
        uint32_t a[16];
        ld_act_block(xs, nblk, b, a);
        float sg, su;
        e8m0x2_to_f32(U.sg[q], U.su[q], sg, su);
        acc[s] = fmaf(block_dot(a, U.g[q]), sg, acc[s]);
        acc[SPW + s] = fmaf(block_dot(a, U.u[q]), su, acc[SPW + s]);
      }
    }
  };

  constexpr int kUnits = SPW * NSEG;
  // the first unit's codes are requested before the activation prologue
  GateUpUnit U;
  load_unit(0, 0, U);
  const int sigma = stage_activations(x + (size_t)t * H, 1, H, xs, red);
  const float unscale = exp2i(-sigma);
#pragma unroll
  for (int u = 0; u < kUnits; ++u) {
    compute_unit(u / NSEG, u % NSEG, U);
    if (u + 1 < kUnits) load_unit((u + 1) / NSEG, (u + 1) % NSEG, U);
  }

  // lane l now holds the total of value l >> (4 - log2 SPW): gate sums in
  // lanes 0..15, the matching up sums 16 lanes higher
  const float tot = warp_sum_transposed<2 * SPW>(acc);
  const float up_tot = __shfl_down_sync(0xFFFFFFFFu, tot, 16);
  constexpr int kLanesPerSlot = 16 / SPW;
  const int s = lane / kLanesPerSlot;
  const int e = __shfl_sync(0xFFFFFFFFu, e_lane, s & (SPW - 1));
  if (lane < 16 && lane % kLanesPerSlot == 0 && s < nslots) {
    const size_t out = ((size_t)t * top_k + j0 + s) * I + n;
    if (e >= 0 && e < E) {
      const float g = tot * unscale, uu = up_tot * unscale;
      const float sl = g / (1.0f + expf(-g));
      const __nv_bfloat16 hv = __float2bfloat16_rn(sl * uu);
      h[out] = *reinterpret_cast<const uint16_t*>(&hv);
    } else {
      h[out] = 0;
      flag_invalid(err);
    }
  }
}

template <int SPW, int NSEG, bool FULL, int KH, int MINB = 3>
moe_status launch_gate_up(const moe_shape* s, const moe_weights* w, const uint16_t* x,
                          const int32_t* ids, int32_t B, uint16_t* h, int32_t* err,
                          cudaStream_t st, RouteArgs route) {
  const size_t smem = (size_t)s->H * 2;
  moe_status rc = allow_smem(moe_gate_up_kernel<SPW, NSEG, FULL, KH, MINB>, smem);
  if (rc != MOE_OK) return rc;
  const int groups = (s->top_k + SPW - 1) / SPW;
  const dim3 grid((unsigned)(B * groups), (unsigned)(s->I / kWarpsPerCta));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = route.dependent ? 1 : 0;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, moe_gate_up_kernel<SPW, NSEG, FULL, KH, MINB>,
                                           w->gu_codes, w->gu_scales, x, ids, h, err, s->H,
                                           s->I, s->E, s->top_k, route);
  if (e != cudaSuccess) {
    set_error("moe_gate_up launch", e);
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

}  // namespace
}  // namespace wd
