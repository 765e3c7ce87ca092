// moe_down: the second kernel of the layer and its launcher.
#include "wd_device.cuh"

namespace wd {
namespace {

// --------------------------------------------------------------- moe_down --
// grid.x = B (token), grid.y = H / (8*OPW) (output block); 8 warps, warp w owns
// outputs o0 .. o0+OPW-1 with o0 = (8*blockIdx.y + w) * OPW. Dynamic shared
// memory: the token's top_k intermediates as scaled f16 (top_k * I), plus
// the token's ids and routing weights.
//
// A warp's top_k * I/32 (slot, block) units are spread over its lanes; every
// unit multiplies one block of the intermediate (read once from shared memory)
// with the same block of the OPW down rows, and adds partial * scale * w[slot]
// into the lane's OPW FP32 accumulators -- the routing weight is folded into
// the sum, so no per-expert output exists.

template <int OPW>
struct DownUnit {
  Codes32 c[OPW];
  uint32_t s[OPW];
};

// The unit's OPW block scales as FP32, two per hardware conversion.
template <int OPW>
__device__ __forceinline__ void unit_scales(const DownUnit<OPW>& U, float (&sc)[OPW]) {
  if constexpr (OPW == 1) {
    float unused;
    e8m0x2_to_f32(U.s[0], 0u, sc[0], unused);
  } else {
#pragma unroll
    for (int r = 0; r < OPW; r += 2) e8m0x2_to_f32(U.s[r], U.s[r + 1], sc[r], sc[r + 1]);
  }
}

// UPL: units each lane requests at once. When the whole grid fits on the GPU
// in one wave (small batches), a lane with OPW < 8 outputs has registers to
// keep UPL = 8 / OPW of its (slot, block) units in flight instead of one HBM
// round trip each.
// KI: the row length I fixed at compile time (0: taken from the argument). With
// it the row strides are constants the loads take as immediates, and the
// (slot, block) advance divides by a constant.
template <int OPW, int UPL, int KI>
__global__ void __launch_bounds__(kThreads, (OPW * UPL >= 8) ? 2 : 3)
    moe_down_kernel(const uint8_t* __restrict__ d_codes, const uint8_t* __restrict__ d_scales,
                    const uint16_t* __restrict__ h, const int32_t* __restrict__ ids,
                    const float* __restrict__ wts, float* __restrict__ y,
                    int32_t* __restrict__ err, int H, int I_arg, int E, int top_k,
                    const float* __restrict__ logits) {
  const int I = KI ? KI : I_arg;
  extern __shared__ uint4 dyn[];
  __shared__ float red[kWarpsPerCta];
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x;
  const int o0 = (blockIdx.y * kWarpsPerCta + (threadIdx.x >> 5)) * OPW;
  const int nblk = I >> 5;
  uint4* hs = dyn;                                                      // top_k*I/8 uint4
  int* s_ids = reinterpret_cast<int*>(dyn + (size_t)top_k * (I >> 3));  // top_k
  float* s_w = reinterpret_cast<float*>(s_ids + top_k);                 // top_k

  const int units = top_k * nblk;
  float acc[OPW];
#pragma unroll
  for (int r = 0; r < OPW; ++r) acc[r] = 0.0f;
  bool bad = false;

  auto load_unit = [&](int e, int bb, DownUnit<OPW>& U) {
    if (e < 0 || e >= E) return;
#pragma unroll
    for (int r = 0; r < OPW; ++r) {
      const size_t row = (size_t)e * H + o0 + r;
      U.c[r] = ld_codes32(d_codes + row * I + (size_t)bb * 32);
      U.s[r] = __ldg(d_scales + row * nblk + bb);
    }
  };
  auto compute_unit = [&](int jj, int bb, const DownUnit<OPW>& U) {
    const int e = s_ids[jj];
    if (e < 0 || e >= E) {
      bad = true;
      return;
    }
    const float wj = s_w[jj];
    uint32_t a[16];
    ld_act_block(hs + (size_t)jj * (I >> 3), nblk, bb, a);
    float sc[OPW];
    unit_scales(U, sc);
#pragma unroll
    for (int r = 0; r < OPW; ++r) acc[r] = fmaf(block_dot(a, U.c[r]), sc[r] * wj, acc[r]);
  };
  // (slot, block) of a unit, advanced by `step` units
  auto advance = [&](int& jj, int& bb, int step) {
    bb += step;
    const int q = bb / nblk;
    jj += q;
    bb -= q * nblk;
  };

  // This lane's units are u = lane + 32*(q + UPL*i); a batch holds q < UPL.
  int jj[UPL], bb[UPL];
  jj[0] = lane / nblk;
  bb[0] = lane - jj[0] * nblk;
#pragma unroll
  for (int q = 1; q < UPL; ++q) {
    jj[q] = jj[q - 1];
    bb[q] = bb[q - 1];
    advance(jj[q], bb[q], 32);
  }
  DownUnit<OPW> U[UPL];

  // The ids, routing weights and down weights are inputs of the layer, not
  // produced by moe_gate_up: the first batch is requested before waiting for
  // the intermediate.
  if (logits) {  // route the token here, from its logits (same result as gate_up)
    int rid;
    float rw;
    warp_route(logits + (size_t)t * E, E, top_k, rid, rw);
#pragma unroll
    for (int q = 0; q < UPL; ++q) {
      const int e = __shfl_sync(0xFFFFFFFFu, rid, jj[q] < top_k ? jj[q] : 0);
      if (lane + 32 * q < units) load_unit(e, bb[q], U[q]);
    }
    if (threadIdx.x < top_k) {
      s_ids[threadIdx.x] = rid;
      s_w[threadIdx.x] = rw;
    }
  } else {
#pragma unroll
    for (int q = 0; q < UPL; ++q)
      if (lane + 32 * q < units) load_unit(__ldg(ids + (size_t)t * top_k + jj[q]), bb[q], U[q]);
    for (int j = threadIdx.x; j < top_k; j += kThreads) {
      s_ids[j] = __ldg(ids + (size_t)t * top_k + j);
      s_w[j] = __ldg(wts + (size_t)t * top_k + j);
    }
  }
  wait_prerequisite();  // the intermediate h is complete from here on
  const int sigma = stage_activations<true>(h + (size_t)t * top_k * I, top_k, I, hs, red);
  const float unscale = exp2i(-sigma);

  if constexpr (OPW == 8 && UPL == 1) {
    // Two halves of 4 rows: as soon as a half of this unit has been used, its
    // registers are refilled with the same rows of the lane's next unit, so the
    // next unit's first half is in flight while the second half is computed.
    // (Eight single-row refills were 2x slower -- a warp has too few load
    // scoreboards for that many staggered groups -- and four pairs slower than
    // two halves. Q30 B=32: 50.1 -> 44.1 us; the same for 4 outputs per warp
    // was mixed across shapes.)
    for (int u0 = lane; u0 < units; u0 += 32) {
      int jn = jj[0], bn = bb[0];
      advance(jn, bn, 32);
      const int en = (u0 + 32 < units) ? s_ids[jn] : -1;
      const bool refill = en >= 0 && en < E;
      const int e = s_ids[jj[0]];
      const bool ok = e >= 0 && e < E;
      if (!ok) bad = true;
      const float wj = s_w[jj[0]];
      uint32_t a[16];
      ld_act_block(hs + (size_t)jj[0] * (I >> 3), nblk, bb[0], a);
      float sc[8];
      unit_scales(U[0], sc);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
#pragma unroll
        for (int r = 4 * half; r < 4 * half + 4; ++r)
          if (ok) acc[r] = fmaf(block_dot(a, U[0].c[r]), sc[r] * wj, acc[r]);
        if (refill) {
          const size_t row0 = (size_t)en * H + o0;
#pragma unroll
          for (int r = 4 * half; r < 4 * half + 4; ++r) {
            U[0].c[r] = ld_codes32(d_codes + (row0 + r) * I + (size_t)bn * 32);
            U[0].s[r] = __ldg(d_scales + (row0 + r) * nblk + bn);
          }
        }
      }
      jj[0] = jn;
      bb[0] = bn;
    }
  } else {
    for (int u0 = lane; u0 < units; u0 += 32 * UPL) {
#pragma unroll
      for (int q = 0; q < UPL; ++q)
        if (u0 + 32 * q < units) compute_unit(jj[q], bb[q], U[q]);
#pragma unroll
      for (int q = 0; q < UPL; ++q) {
        advance(jj[q], bb[q], 32 * UPL);
        if (u0 + 32 * (UPL + q) < units) load_unit(s_ids[jj[q]], bb[q], U[q]);
      }
    }
  }
  // lane l holds the total of output l / (32 / OPW)
  const float tot = warp_sum_transposed<OPW>(acc) * unscale;
  if (bad) flag_invalid(err);
  if (lane % (32 / OPW) == 0) y[(size_t)t * H + o0 + lane / (32 / OPW)] = tot;
}

// Outputs per warp of moe_down beyond the single-wave small batches: 8 for
// rows of at most 1536 elements, else as many as keep at least kMinCtasPerSm
// CTAs per SM. Measured on GB300 (in the layer, CUDA graph): Q30 B=16 39.5 ->
// 31.1 us against 2 outputs per warp; Qwen-3-235B-A22B B=8 167.8 -> 154.4 us
// against 2, even with 4 at 16 and 20 tokens; for the 2048-element rows of
// the DeepSeek-V3 shape 8 was up to 0.7 % slower than 4 at 8-40 tokens.
// A CTA covers 8 * OPW outputs, so OPW = 8 needs H % 64 == 0 (H % 32 == 0 is
// enough for the others).
int pick_opw(int B, int H, int I, int sms) {
  if (H % (kWarpsPerCta * 8) == 0 && I <= 1536) return 8;
  const int opws[3] = {4, 2, 1};
  for (int v : opws) {
    const int64_t ctas = (int64_t)B * (H / (kWarpsPerCta * v));
    if (ctas >= (int64_t)kMinCtasPerSm * sms) return v;
  }
  return 1;
}

template <int OPW, int UPL, int KI>
moe_status launch_down_ki(const moe_shape* s, const moe_weights* w, const uint16_t* h,
                          const int32_t* ids, const float* wts, int32_t B, float* y, int32_t* err,
                          cudaStream_t st, bool dependent, const float* logits) {
  const size_t smem = (size_t)s->top_k * s->I * 2 + (size_t)s->top_k * 8;
  moe_status rc = allow_smem(moe_down_kernel<OPW, UPL, KI>, smem);
  if (rc != MOE_OK) return rc;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)B, (unsigned)(s->H / (kWarpsPerCta * OPW)));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 1 : 0;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, moe_down_kernel<OPW, UPL, KI>, w->d_codes,
                                           w->d_scales, h, ids, wts, y, err, s->H, s->I, s->E,
                                           s->top_k, logits);
  if (e != cudaSuccess) {
    set_error("moe_down launch", e);
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

// Row lengths with their own compiled kernel: the intermediate sizes of the
// Qwen3-30B-A3B-, Qwen3-235B-A22B- and DeepSeek-V3-shaped layers; every other
// I runs the kernel that reads I at run time.
template <int OPW, int UPL>
moe_status launch_down(const moe_shape* s, const moe_weights* w, const uint16_t* h,
                       const int32_t* ids, const float* wts, int32_t B, float* y, int32_t* err,
                       cudaStream_t st, bool dependent, const float* logits) {
  if (s->I == 768)
    return launch_down_ki<OPW, UPL, 768>(s, w, h, ids, wts, B, y, err, st, dependent, logits);
  if (s->I == 1536)
    return launch_down_ki<OPW, UPL, 1536>(s, w, h, ids, wts, B, y, err, st, dependent, logits);
  if (s->I == 2048)
    return launch_down_ki<OPW, UPL, 2048>(s, w, h, ids, wts, B, y, err, st, dependent, logits);
  return launch_down_ki<OPW, UPL, 0>(s, w, h, ids, wts, B, y, err, st, dependent, logits);
}

}  // namespace

moe_status launch_down_kernels(const moe_shape* s, const moe_weights* w, const uint16_t* h,
                               const int32_t* ids, const float* wts, int32_t B, float* y,
                               int32_t* err, cudaStream_t st, bool dependent,
                               const float* logits) {
  // Small batches: the fewest outputs per warp (OPW) that make the grid a
  // single wave at 2 CTAs per SM, each lane keeping 8 / OPW units in flight.
  // Fewer, fuller CTAs stage each token's intermediate fewer times and need
  // fewer round trips per lane than one-output warps (Q30 B=8: 32.6 -> 18.5 us).
  const int64_t ctas_opw1 = (int64_t)B * (s->H / kWarpsPerCta);
  const int64_t wave = 2 * (int64_t)sm_count();
  if (ctas_opw1 <= wave)
    return launch_down<1, 8>(s, w, h, ids, wts, B, y, err, st, dependent, logits);
  if (ctas_opw1 / 2 <= wave)
    return launch_down<2, 4>(s, w, h, ids, wts, B, y, err, st, dependent, logits);
  if (ctas_opw1 / 4 <= wave)
    return launch_down<4, 2>(s, w, h, ids, wts, B, y, err, st, dependent, logits);
  if (s->H % (kWarpsPerCta * 8) == 0 && ctas_opw1 / 8 <= wave)
    return launch_down<8, 1>(s, w, h, ids, wts, B, y, err, st, dependent, logits);
  switch (pick_opw(B, s->H, s->I, sm_count())) {
    case 8: return launch_down<8, 1>(s, w, h, ids, wts, B, y, err, st, dependent, logits);
    case 4: return launch_down<4, 1>(s, w, h, ids, wts, B, y, err, st, dependent, logits);
    case 2: return launch_down<2, 1>(s, w, h, ids, wts, B, y, err, st, dependent, logits);
    default: return launch_down<1, 1>(s, w, h, ids, wts, B, y, err, st, dependent, logits);
  }
}

}  // namespace wd
