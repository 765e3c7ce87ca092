// GB300 (sm_103a) kernels and C-ABI launchers of the output-centric
// ("warp decode") MoE decode layer.
//
// Method: "Better MoE model inference with warp decode" (Key claims
// [§Reorganized parallelism], [§How the two kernels work], [§Warp Independence];
// Method) and the sd114.wiki "Warp Decode" page (section
// 技术原理：两个 Kernel 搞定一切): every warp owns output scalars, streams the
// weight rows it needs from HBM into private FP32 accumulators, and finishes
// with a __shfl_xor_sync butterfly; no cross-warp reduction exists.
//
// GB300 design (numbers from measurements on this part):
//  * Instruction budget. FP32 FFMA and the mixed-precision fma.rn.f32.f16 issue
//    at full rate, while every integer, logic and conversion instruction
//    (LOP3, SHF, PRMT, cvt) issues at half rate. The inner loop is therefore
//      hardware cvt e4m3x2 -> f16x2        (0.5 half-rate instr / weight)
//      fma.rn.f32.f16 activation x weight  (1 full-rate instr / weight)
//    The product of an f16 activation and an E4M3 weight is exact and is
//    accumulated in FP32, as in the pages' FP32-accumulator design.
//  * Activations as f16. The BF16 activation row (x for gate/up, the routed
//    intermediate for down) is converted once per CTA into shared memory as
//    f16 after a power-of-two scale 2^sigma that puts its largest magnitude in
//    [2^14, 2^15); results are multiplied back by 2^-sigma. Every BF16 value
//    within 2^29 of the row's maximum is represented exactly; smaller ones are
//    rounded to a multiple of 2^-24 * 2^-sigma (far below FP32 accumulation
//    error). The f16 copy is laid out [4][blocks][16 B] so that 32 lanes
//    reading 16 B each hit 32 distinct banks.
//  * Memory. Each lane owns whole 32-element MXFP8 blocks (one E8M0 scale per
//    block): one 256-bit load of 32 codes per block, so a warp-wide load reads
//    1 KB of one row contiguously. Weight loads bypass L1 allocation; reuse of
//    a row by several tokens happens in L2, which the grid order makes likely
//    (neuron/output block is the slow grid axis, tokens the fast one).
//  * Latency is hidden by occupancy: both kernels are kept at <= 80 registers
//    so that 3 CTAs (24 warps) fit on an SM. (Holding a second unit of codes in
//    registers to prefetch it, or staging codes through a cp.async ring in
//    shared memory, both measured slower on this part.) moe_gate_up warps loop
//    over several routed slots of one token; moe_down warps own several
//    outputs that share one read of the intermediate from shared memory.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <mutex>

#include "warp_decode.h"

namespace {

constexpr int kWarpsPerCta = 8;  // 8 warps per CTA, as the pages give for moe_gate_up
constexpr int kThreads = kWarpsPerCta * 32;
constexpr int kSegBlocksPerLane = 2;               // gate/up: 32-element blocks per lane per unit
constexpr int kSegBlocks = 32 * kSegBlocksPerLane;  // blocks of one row per unit (2048 elements)
constexpr int kMinCtas = 8 * 152;                  // enough CTAs to fill 152 SMs several times

// ---------------------------------------------------------------- loads ----

struct Codes32 {
  uint32_t w[8];  // 32 E4M3 codes, element 4i+b in byte b of w[i]
};

// One 32-element block of codes: a 256-bit load that does not allocate in L1.
__device__ __forceinline__ Codes32 ld_codes32(const uint8_t* p) {
  Codes32 c;
  asm("ld.global.nc.L1::no_allocate.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(c.w[0]), "=r"(c.w[1]), "=r"(c.w[2]), "=r"(c.w[3]), "=r"(c.w[4]), "=r"(c.w[5]),
        "=r"(c.w[6]), "=r"(c.w[7])
      : "l"(p));
  return c;
}

__device__ __forceinline__ uint4 ld_cached16(const void* p) {
  uint4 r;
  asm("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

// ---------------------------------------------------------------- decode ---

// E8M0 scale code -> 2^(s-127) as FP32 (0 -> 2^-127, a subnormal; 255 -> NaN).
__device__ __forceinline__ float e8m0_to_f32(uint32_t s) {
  uint32_t bits = s << 23;
  bits = (s == 0u) ? 0x00400000u : bits;
  bits = (s == 255u) ? 0x7FC00000u : bits;
  return __uint_as_float(bits);
}

// 2^e for e in [-126, 127], exact.
__device__ __forceinline__ float exp2i(int e) { return __uint_as_float((uint32_t)(e + 127) << 23); }

// Four E4M3 codes (one word) -> two f16x2 words, exact (hardware conversion).
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{.reg .b16 a, b;\n\t"
      "mov.b32 {a, b}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, a;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// c + a.lo*b.lo + a.hi*b.hi with f16 operands, exact products, FP32 sums.
__device__ __forceinline__ float fma2_f16(uint32_t a, uint32_t b, float c) {
  asm("{.reg .b16 al, ah, bl, bh;\n\t"
      "mov.b32 {al, ah}, %1;\n\t"
      "mov.b32 {bl, bh}, %2;\n\t"
      "fma.rn.f32.f16 %0, al, bl, %0;\n\t"
      "fma.rn.f32.f16 %0, ah, bh, %0;\n\t}"
      : "+f"(c)
      : "r"(a), "r"(b));
  return c;
}

// sum over one 32-element block: f16 activations a[16 words] x E4M3 codes.
__device__ __forceinline__ float block_dot(const uint32_t (&a)[16], const Codes32& c) {
  float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint32_t lo, hi;
    e4m3x4_to_f16x4(c.w[i], lo, hi);
    s0 = fma2_f16(a[2 * i], lo, s0);
    s1 = fma2_f16(a[2 * i + 1], hi, s1);
  }
  return s0 + s1;
}

// 16 f16 activations of block b from the swizzled shared copy ([4][nblk] x 16 B).
__device__ __forceinline__ void ld_act_block(const uint4* act, int nblk, int b, uint32_t (&a)[16]) {
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const uint4 v = act[m * nblk + b];
    a[4 * m + 0] = v.x;
    a[4 * m + 1] = v.y;
    a[4 * m + 2] = v.z;
    a[4 * m + 3] = v.w;
  }
}

// ------------------------------------------------------- activation prologue
// BF16 row(s) in global memory -> f16 x 2^sigma in shared memory, sigma chosen
// per row group so that the largest magnitude lands in [2^14, 2^15).

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ float absmax8(const uint4& v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w[i])), fabsf(bf16_hi(w[i]))));
  return m;
}

__device__ __forceinline__ uint4 to_f16x8(const uint4& v, float scale) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 h = __floats2half2_rn(bf16_lo(w[i]) * scale, bf16_hi(w[i]) * scale);
    o[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, m));
  return v;
}

// sigma such that m * 2^sigma is in [2^14, 2^15); 0 for m = 0, inf or NaN.
__device__ __forceinline__ int pow2_shift_for(float m) {
  if (!(m > 0.0f) || isinf(m)) return 0;
  int ex;
  frexpf(m, &ex);  // m = f * 2^ex, f in [0.5, 1)
  return min(126, max(-126, 15 - ex));
}

// Convert `rows` BF16 rows of `len` elements (row r at src + r*len) into the
// swizzled f16 layout dst[r][4][len/32] (uint4 units) with one shared scale.
// Returns sigma. Must be called by all threads of the CTA.
__device__ int stage_activations(const uint16_t* __restrict__ src, int rows, int len,
                                 uint4* dst, float* red) {
  const int pieces_per_row = len >> 3;  // 16-byte pieces (8 elements)
  const int pieces = rows * pieces_per_row;
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
  float m = 0.0f;
  for (int p = threadIdx.x; p < pieces; p += kThreads) m = fmaxf(m, absmax8(ld_cached16(s4 + p)));
  m = warp_max(m);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  m = red[0];
#pragma unroll
  for (int i = 1; i < kWarpsPerCta; ++i) m = fmaxf(m, red[i]);
  const int sigma = pow2_shift_for(m);
  const float up = exp2i(sigma);
  const int nblk = len >> 5;
  for (int p = threadIdx.x; p < pieces; p += kThreads) {
    const int r = p / pieces_per_row, q = p - r * pieces_per_row;
    dst[r * pieces_per_row + (q & 3) * nblk + (q >> 2)] = to_f16x8(ld_cached16(s4 + p), up);
  }
  __syncthreads();
  return sigma;
}

// Programmatic dependent launch (moe_layer launches moe_down as a dependent of
// moe_gate_up). launch_dependents lets the dependent grid be scheduled once
// every CTA of this grid has issued it; wait_prerequisite blocks until the
// prerequisite grid has completed and its writes are visible (it returns at
// once when the kernel was not launched as a dependent). Both are hardware
// grid dependencies, not spins on memory.
__device__ __forceinline__ void launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void wait_prerequisite() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void flag_invalid(int32_t* err) {
  if (err) atomicOr(err, 1);
}

// ------------------------------------------------------------------ router --
// Routing of one token from its router logits (the step in front of the layer:
// "Better MoE model inference with warp decode", Method: each token goes to
// the top-k of E experts). The renormalised top-k of softmax(logits) equals a
// softmax over the k largest logits, so the experts are chosen on the logits
// themselves (largest first, ties to the lower index) and
//   w_j = exp(l_j - l_max) / sum over the chosen i of exp(l_i - l_max).
// One warp; lane j < top_k receives the j-th choice. E <= 256, top_k <= 32,
// logits finite.
constexpr int kRouteMaxE = 256;

struct RouteArgs {
  const float* logits;  // [B][E], or nullptr: the ids/wts arrays are the routing
  int32_t* ids_out;     // routing chosen by the kernel, written if non-null
  float* w_out;
};

__device__ __noinline__ void warp_route(const float* __restrict__ row, int E, int top_k,
                                           int& id, float& weight) {
  constexpr int kPer = kRouteMaxE / 32;
  const int lane = threadIdx.x & 31;
  float v[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) v[i] = (lane + 32 * i < E) ? __ldg(row + lane + 32 * i) : 0.0f;
  uint32_t open = 0;  // bit i: candidate lane + 32 i still available
#pragma unroll
  for (int i = 0; i < kPer; ++i)
    if (lane + 32 * i < E) open |= 1u << i;
  id = -1;
  float mine = 0.0f, lmax = 0.0f;
  for (int j = 0; j < top_k; ++j) {
    float bv = 0.0f;
    int be = 0x7FFFFFFF;  // none
#pragma unroll
    for (int i = 0; i < kPer; ++i)
      if (((open >> i) & 1u) && (be == 0x7FFFFFFF || v[i] > bv)) {
        bv = v[i];
        be = lane + 32 * i;
      }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) {
      const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, m);
      const int oe = __shfl_xor_sync(0xFFFFFFFFu, be, m);
      if (oe != 0x7FFFFFFF && (be == 0x7FFFFFFF || ov > bv || (ov == bv && oe < be))) {
        bv = ov;
        be = oe;
      }
    }
    if ((be & 31) == lane) open &= ~(1u << (be >> 5));
    if (lane == j) {
      id = be;
      mine = bv;
    }
    if (j == 0) lmax = bv;
  }
  float ex = (lane < top_k) ? expf(mine - lmax) : 0.0f;
  float sum = ex;
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, m);
  weight = ex / sum;
}

// moe_route: one warp per token.
__global__ void __launch_bounds__(kThreads)
    moe_route_kernel(const float* __restrict__ logits, int32_t* __restrict__ ids,
                     float* __restrict__ wts, int B, int E, int top_k) {
  const int t = blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  if (t >= B) return;
  const int lane = threadIdx.x & 31;
  int id;
  float w;
  warp_route(logits + (size_t)t * E, E, top_k, id, w);
  if (lane < top_k) {
    ids[(size_t)t * top_k + lane] = id;
    wts[(size_t)t * top_k + lane] = w;
  }
}

// Sum each of the V (a power of two, <= 32) values of v over the 32 lanes of
// the warp with one transposing butterfly: at every step a lane keeps half
// of its values and receives its partner's partial sums of that half, so the
// values are reduced together in V-1 + (5 - log2 V) shuffles instead of
// V*5. Afterwards lane l holds the total of value index l >> (5 - log2 V).
template <int V>
__device__ __forceinline__ float warp_sum_transposed(float (&v)[V]) {
  static_assert(V == 1 || V == 2 || V == 4 || V == 8 || V == 16 || V == 32, "V: power of two");
  constexpr int L = V == 1 ? 0 : V == 2 ? 1 : V == 4 ? 2 : V == 8 ? 3 : V == 16 ? 4 : 5;
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int k = 0; k < L; ++k) {
    const int m = 16 >> k;
    const int half = V >> (k + 1);
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = upper ? v[i] : v[i + half];
      const float keep = upper ? v[i + half] : v[i];
      v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, m);
    }
  }
  float r = v[0];
#pragma unroll
  for (int m = 16 >> L; m >= 1; m >>= 1) r += __shfl_xor_sync(0xFFFFFFFFu, r, m);
  return r;
}

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
template <int SPW, int NSEG, bool FULL>
__global__ void __launch_bounds__(kThreads, 3)
    moe_gate_up_kernel(const uint8_t* __restrict__ gu_codes,
                       const uint8_t* __restrict__ gu_scales,
                       const uint16_t* __restrict__ x, const int32_t* __restrict__ ids,
                       uint16_t* __restrict__ h, int32_t* __restrict__ err, int H, int I,
                       int E, int top_k, RouteArgs route) {
  extern __shared__ uint4 xs[];
  __shared__ float red[kWarpsPerCta];
  const int lane = threadIdx.x & 31;
  const int groups = (top_k + SPW - 1) / SPW;
  const int t = blockIdx.x / groups;
  const int j0 = (blockIdx.x - t * groups) * SPW;
  const int n = blockIdx.y * kWarpsPerCta + (threadIdx.x >> 5);
  const int nblk = H >> 5;
  const int nslots = min(SPW, top_k - j0);

  launch_dependents();

  // lane s < nslots holds the expert id of slot s; -1 marks "no slot"
  int e_lane;
  if (route.logits) {  // route the token here, from its logits
    int rid;
    float rw;
    warp_route(route.logits + (size_t)t * E, E, top_k, rid, rw);
    e_lane = __shfl_sync(0xFFFFFFFFu, rid, lane < nslots ? j0 + lane : 0);
    if (lane >= nslots) e_lane = -1;
    if (route.ids_out && j0 == 0 && blockIdx.y == 0 && threadIdx.x < top_k) {
      route.ids_out[(size_t)t * top_k + lane] = rid;
      route.w_out[(size_t)t * top_k + lane] = rw;
    }
  } else {
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
        acc[s] = fmaf(block_dot(a, U.g[q]), e8m0_to_f32(U.sg[q]), acc[s]);
        acc[SPW + s] = fmaf(block_dot(a, U.u[q]), e8m0_to_f32(U.su[q]), acc[SPW + s]);
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

// UPL: units each lane requests at once. When the whole grid fits on the GPU
// in one wave (small batches), a lane with one output has registers to keep
// UPL of its (slot, block) units in flight instead of one HBM round trip each.
template <int OPW, int UPL>
__global__ void __launch_bounds__(kThreads, (OPW * UPL >= 8) ? 2 : 3)
    moe_down_kernel(const uint8_t* __restrict__ d_codes, const uint8_t* __restrict__ d_scales,
                    const uint16_t* __restrict__ h, const int32_t* __restrict__ ids,
                    const float* __restrict__ wts, float* __restrict__ y,
                    int32_t* __restrict__ err, int H, int I, int E, int top_k,
                    const float* __restrict__ logits) {
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
#pragma unroll
    for (int r = 0; r < OPW; ++r)
      acc[r] = fmaf(block_dot(a, U.c[r]), e8m0_to_f32(U.s[r]) * wj, acc[r]);
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
  const int sigma = stage_activations(h + (size_t)t * top_k * I, top_k, I, hs, red);
  const float unscale = exp2i(-sigma);

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
  // lane l holds the total of output l / (32 / OPW)
  const float tot = warp_sum_transposed<OPW>(acc) * unscale;
  if (bad) flag_invalid(err);
  if (lane % (32 / OPW) == 0) y[(size_t)t * H + o0 + lane / (32 / OPW)] = tot;
}

// ------------------------------------------------------------- host side ---

thread_local char g_last_error[256] = "";

void set_error(const char* what, cudaError_t e) {
  snprintf(g_last_error, sizeof(g_last_error), "%s: %s", what, cudaGetErrorString(e));
}

void set_error_msg(const char* msg) { snprintf(g_last_error, sizeof(g_last_error), "%s", msg); }

bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p % a) == 0; }

moe_status check_shape(const moe_shape* s, int32_t B) {
  if (!s) return MOE_ERR_NULL;
  if (s->H <= 0 || s->I <= 0 || s->E <= 0 || s->top_k <= 0 || s->top_k > s->E || B < 0 ||
      s->H % 32 || s->I % 32) {
    set_error_msg("shape: need H%32==0, I%32==0, E>=1, 1<=top_k<=E, B>=0");
    return MOE_ERR_SHAPE;
  }
  if (s->H > 8192) {
    set_error_msg("shape: H above 8192 is not supported");
    return MOE_ERR_SHAPE;
  }
  // grid limits: pairs on grid.x (<= 2^31-1), neuron/output blocks on grid.y (<= 65535)
  if ((int64_t)B * s->top_k > 0x7FFFFFFF || (s->I + kWarpsPerCta - 1) / kWarpsPerCta > 65535 ||
      (s->H + kWarpsPerCta - 1) / kWarpsPerCta > 65535) {
    set_error_msg("shape: grid dimensions exceed CUDA limits");
    return MOE_ERR_SHAPE;
  }
  return MOE_OK;
}

moe_status check_weights(const moe_weights* w, bool gate_up, bool down) {
  if (!w) return MOE_ERR_NULL;
  if ((gate_up && (!w->gu_codes || !w->gu_scales)) || (down && (!w->d_codes || !w->d_scales)))
    return MOE_ERR_NULL;
  if ((gate_up && !aligned(w->gu_codes, 32)) || (down && !aligned(w->d_codes, 32))) {
    set_error_msg("alignment: weight codes must be 32-byte aligned");
    return MOE_ERR_ALIGN;
  }
  return MOE_OK;
}

constexpr size_t kMaxDynSmem = 227 * 1024;

// Opt a kernel into more than the default 48 KB of dynamic shared memory.
template <typename K>
moe_status allow_smem(K kernel, size_t bytes) {
  if (bytes > kMaxDynSmem) {
    set_error_msg("shape: activation row does not fit in shared memory");
    return MOE_ERR_UNSUPPORTED;
  }
  if (bytes > 48 * 1024) {
    const cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) {
      set_error("cudaFuncSetAttribute", e);
      return MOE_ERR_CUDA;
    }
  }
  return MOE_OK;
}

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

// Outputs per warp of moe_down: 8 for rows of at most 1024 elements when at
// least 6 CTAs per SM remain (measured faster there), else as many as keep
// at least kMinCtas CTAs.
int pick_opw(int B, int H, int I) {
  if (I <= 1024 && (int64_t)B * (H / (kWarpsPerCta * 8)) >= 6 * 152) return 8;
  const int opws[3] = {4, 2, 1};
  for (int v : opws) {
    const int64_t ctas = (int64_t)B * (H / (kWarpsPerCta * v));
    if (ctas >= kMinCtas) return v;
  }
  return 1;
}

template <int SPW, int NSEG, bool FULL>
moe_status launch_gate_up(const moe_shape* s, const moe_weights* w, const uint16_t* x,
                          const int32_t* ids, int32_t B, uint16_t* h, int32_t* err,
                          cudaStream_t st, RouteArgs route) {
  const size_t smem = (size_t)s->H * 2;
  moe_status rc = allow_smem(moe_gate_up_kernel<SPW, NSEG, FULL>, smem);
  if (rc != MOE_OK) return rc;
  const int groups = (s->top_k + SPW - 1) / SPW;
  const dim3 grid((unsigned)(B * groups), (unsigned)(s->I / kWarpsPerCta));
  moe_gate_up_kernel<SPW, NSEG, FULL><<<grid, kThreads, smem, st>>>(
      w->gu_codes, w->gu_scales, x, ids, h, err, s->H, s->I, s->E, s->top_k, route);
  return MOE_OK;
}

template <int SPW, int NSEG>
moe_status launch_gate_up_full(const moe_shape* s, const moe_weights* w, const uint16_t* x,
                               const int32_t* ids, int32_t B, uint16_t* h, int32_t* err,
                               cudaStream_t st, RouteArgs route) {
  if ((s->H >> 5) % kSegBlocks == 0)
    return launch_gate_up<SPW, NSEG, true>(s, w, x, ids, B, h, err, st, route);
  return launch_gate_up<SPW, NSEG, false>(s, w, x, ids, B, h, err, st, route);
}

template <int NSEG>
moe_status launch_gate_up_spw(const moe_shape* s, const moe_weights* w, const uint16_t* x,
                              const int32_t* ids, int32_t B, uint16_t* h, int32_t* err,
                              cudaStream_t st, RouteArgs route) {
  switch (pick_spw(B, s->top_k, s->I)) {
    case 8: return launch_gate_up_full<8, NSEG>(s, w, x, ids, B, h, err, st, route);
    case 4: return launch_gate_up_full<4, NSEG>(s, w, x, ids, B, h, err, st, route);
    case 2: return launch_gate_up_full<2, NSEG>(s, w, x, ids, B, h, err, st, route);
    default: return launch_gate_up_full<1, NSEG>(s, w, x, ids, B, h, err, st, route);
  }
}

// dependent = true launches moe_down as a programmatic dependent of the kernel
// before it on the stream (used by moe_layer, where that kernel is moe_gate_up
// and only h is produced by it).
template <int OPW, int UPL>
moe_status launch_down(const moe_shape* s, const moe_weights* w, const uint16_t* h,
                       const int32_t* ids, const float* wts, int32_t B, float* y, int32_t* err,
                       cudaStream_t st, bool dependent, const float* logits) {
  const size_t smem = (size_t)s->top_k * s->I * 2 + (size_t)s->top_k * 8;
  moe_status rc = allow_smem(moe_down_kernel<OPW, UPL>, smem);
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
  const cudaError_t e = cudaLaunchKernelEx(&cfg, moe_down_kernel<OPW, UPL>, w->d_codes, w->d_scales, h,
                                           ids, wts, y, err, s->H, s->I, s->E, s->top_k, logits);
  if (e != cudaSuccess) {
    set_error("moe_down launch", e);
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}


moe_status launch_status(const char* what) {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error(what, e);
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

// Checks of the routed entry points: the warp router handles E <= 256 and
// top_k <= 32; logits are FP32 [B][E], 4-byte aligned.
moe_status check_route(const moe_shape* s, const float* logits) {
  if (!logits) return MOE_ERR_NULL;
  if (s->E > kRouteMaxE || s->top_k > 32) {
    set_error_msg("routing on the device needs E <= 256 and top_k <= 32");
    return MOE_ERR_UNSUPPORTED;
  }
  if (!aligned(logits, 4)) {
    set_error_msg("alignment: logits need 4 bytes");
    return MOE_ERR_ALIGN;
  }
  return MOE_OK;
}

constexpr RouteArgs kNoRoute = {nullptr, nullptr, nullptr};

moe_status gate_up_impl(const moe_shape* s, const moe_weights* w, const uint16_t* x,
                        const int32_t* ids, int32_t B, uint16_t* h, int32_t* err,
                        cudaStream_t st, RouteArgs route = kNoRoute) {
  moe_status rc = check_shape(s, B);
  if (rc != MOE_OK) return rc;
  if ((rc = check_weights(w, true, false)) != MOE_OK) return rc;
  if (B == 0) return MOE_OK;
  if (!x || (!ids && !route.logits) || !h) return MOE_ERR_NULL;
  if (!aligned(x, 16) || !aligned(h, 16) || !aligned(ids, 4) || !aligned(err, 4)) {
    set_error_msg("alignment: x and h need 16 bytes, ids and err_flag 4");
    return MOE_ERR_ALIGN;
  }
  const int nseg = ((s->H >> 5) + kSegBlocks - 1) / kSegBlocks;  // 2048-element row segments
  if (nseg == 1) rc = launch_gate_up_spw<1>(s, w, x, ids, B, h, err, st, route);
  else if (nseg == 2) rc = launch_gate_up_spw<2>(s, w, x, ids, B, h, err, st, route);
  else rc = launch_gate_up_spw<4>(s, w, x, ids, B, h, err, st, route);
  if (rc != MOE_OK) return rc;
  return launch_status("moe_gate_up launch");
}

moe_status down_impl(const moe_shape* s, const moe_weights* w, const uint16_t* h,
                     const int32_t* ids, const float* wts, int32_t B, float* y, int32_t* err,
                     cudaStream_t st, bool dependent, const float* logits = nullptr) {
  moe_status rc = check_shape(s, B);
  if (rc != MOE_OK) return rc;
  if ((rc = check_weights(w, false, true)) != MOE_OK) return rc;
  if (B == 0) return MOE_OK;
  if (!h || ((!ids || !wts) && !logits) || !y) return MOE_ERR_NULL;
  if (!aligned(h, 16) || !aligned(ids, 4) || !aligned(wts, 4) || !aligned(y, 4) ||
      !aligned(err, 4)) {
    set_error_msg("alignment: h needs 16 bytes, ids/wts/y/err_flag 4");
    return MOE_ERR_ALIGN;
  }
  switch (pick_opw(B, s->H, s->I)) {
    case 8: rc = launch_down<8, 1>(s, w, h, ids, wts, B, y, err, st, dependent, logits); break;
    case 4: rc = launch_down<4, 1>(s, w, h, ids, wts, B, y, err, st, dependent, logits); break;
    case 2: rc = launch_down<2, 1>(s, w, h, ids, wts, B, y, err, st, dependent, logits); break;
    default:
      // one output per warp: batch 8 units per lane when the grid is one wave
      // at 2 CTAs per SM
      if ((int64_t)B * (s->H / kWarpsPerCta) <= 2 * 152)
        rc = launch_down<1, 8>(s, w, h, ids, wts, B, y, err, st, dependent, logits);
      else
        rc = launch_down<1, 1>(s, w, h, ids, wts, B, y, err, st, dependent, logits);
      break;
  }
  if (rc != MOE_OK) return rc;
  return launch_status("moe_down launch");
}

}  // namespace

extern "C" moe_status moe_gate_up(const moe_shape* shape, const moe_weights* w,
                                  const uint16_t* x, const int32_t* ids, int32_t B,
                                  uint16_t* h, int32_t* err_flag, void* stream) {
  return gate_up_impl(shape, w, x, ids, B, h, err_flag, (cudaStream_t)stream);
}

extern "C" moe_status moe_down(const moe_shape* shape, const moe_weights* w, const uint16_t* h,
                               const int32_t* ids, const float* wts, int32_t B, float* y,
                               int32_t* err_flag, void* stream) {
  return down_impl(shape, w, h, ids, wts, B, y, err_flag, (cudaStream_t)stream, false);
}

extern "C" moe_status moe_layer(const moe_shape* shape, const moe_weights* w, const uint16_t* x,
                                const int32_t* ids, const float* wts, int32_t B,
                                uint16_t* h_scratch, float* y, int32_t* err_flag,
                                void* stream) {
  // validate everything before the first launch, so a bad argument launches nothing
  moe_status rc = check_shape(shape, B);
  if (rc != MOE_OK) return rc;
  if ((rc = check_weights(w, true, true)) != MOE_OK) return rc;
  if (B == 0) return MOE_OK;
  if (!x || !ids || !wts || !h_scratch || !y) return MOE_ERR_NULL;
  rc = gate_up_impl(shape, w, x, ids, B, h_scratch, err_flag, (cudaStream_t)stream);
  if (rc != MOE_OK) return rc;
  return down_impl(shape, w, h_scratch, ids, wts, B, y, err_flag, (cudaStream_t)stream, true);
}

extern "C" moe_status moe_route(const moe_shape* shape, const float* logits, int32_t B,
                                int32_t* ids, float* wts, void* stream) {
  moe_status rc = check_shape(shape, B);
  if (rc != MOE_OK) return rc;
  if ((rc = check_route(shape, logits)) != MOE_OK) return rc;
  if (B == 0) return MOE_OK;
  if (!ids || !wts) return MOE_ERR_NULL;
  if (!aligned(ids, 4) || !aligned(wts, 4)) {
    set_error_msg("alignment: ids and wts need 4 bytes");
    return MOE_ERR_ALIGN;
  }
  const unsigned grid = (unsigned)((B + kWarpsPerCta - 1) / kWarpsPerCta);
  moe_route_kernel<<<grid, kThreads, 0, (cudaStream_t)stream>>>(logits, ids, wts, B, shape->E,
                                                               shape->top_k);
  return launch_status("moe_route launch");
}

extern "C" moe_status moe_layer_routed(const moe_shape* shape, const moe_weights* w,
                                       const uint16_t* x, const float* logits, int32_t B,
                                       uint16_t* h_scratch, float* y, int32_t* ids_out,
                                       float* wts_out, int32_t* err_flag, void* stream) {
  moe_status rc = check_shape(shape, B);
  if (rc != MOE_OK) return rc;
  if ((rc = check_weights(w, true, true)) != MOE_OK) return rc;
  if ((rc = check_route(shape, logits)) != MOE_OK) return rc;
  if (B == 0) return MOE_OK;
  if (!x || !h_scratch || !y) return MOE_ERR_NULL;
  if ((ids_out == nullptr) != (wts_out == nullptr)) return MOE_ERR_NULL;
  if (!aligned(ids_out, 4) || !aligned(wts_out, 4)) {
    set_error_msg("alignment: ids_out and wts_out need 4 bytes");
    return MOE_ERR_ALIGN;
  }
  const RouteArgs route = {logits, ids_out, wts_out};
  rc = gate_up_impl(shape, w, x, nullptr, B, h_scratch, err_flag, (cudaStream_t)stream, route);
  if (rc != MOE_OK) return rc;
  return down_impl(shape, w, h_scratch, nullptr, nullptr, B, y, err_flag, (cudaStream_t)stream,
                   true, logits);
}

extern "C" moe_status moe_layer_host(const moe_shape* shape, const moe_weights* w,
                                     const uint16_t* x_host, const int32_t* ids_host,
                                     const float* wts_host, int32_t B, uint16_t* x_dev,
                                     int32_t* ids_dev, float* wts_dev, uint16_t* h_dev,
                                     float* y_dev, float* y_host, int32_t* err_flag,
                                     void* stream) {
  moe_status rc = check_shape(shape, B);
  if (rc != MOE_OK) return rc;
  if ((rc = check_weights(w, true, true)) != MOE_OK) return rc;
  if (B == 0) return MOE_OK;
  if (!x_host || !ids_host || !wts_host || !y_host || !x_dev || !ids_dev || !wts_dev || !h_dev ||
      !y_dev)
    return MOE_ERR_NULL;
  if (!aligned(x_dev, 16) || !aligned(h_dev, 16) || !aligned(ids_dev, 4) ||
      !aligned(wts_dev, 4) || !aligned(y_dev, 4)) {
    set_error_msg("alignment: x_dev and h_dev need 16 bytes, others 4");
    return MOE_ERR_ALIGN;
  }
  cudaStream_t st = (cudaStream_t)stream;
  const size_t nx = (size_t)B * shape->H, nk = (size_t)B * shape->top_k;
  cudaError_t e;
  if ((e = cudaMemcpyAsync(x_dev, x_host, nx * 2, cudaMemcpyHostToDevice, st)) != cudaSuccess ||
      (e = cudaMemcpyAsync(ids_dev, ids_host, nk * 4, cudaMemcpyHostToDevice, st)) != cudaSuccess ||
      (e = cudaMemcpyAsync(wts_dev, wts_host, nk * 4, cudaMemcpyHostToDevice, st)) !=
          cudaSuccess) {
    set_error("moe_layer_host: host->device copy", e);
    return MOE_ERR_CUDA;
  }
  rc = moe_layer(shape, w, x_dev, ids_dev, wts_dev, B, h_dev, y_dev, err_flag, stream);
  if (rc != MOE_OK) return rc;
  if ((e = cudaMemcpyAsync(y_host, y_dev, nx * 4, cudaMemcpyDeviceToHost, st)) != cudaSuccess) {
    set_error("moe_layer_host: device->host copy", e);
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

extern "C" const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_NULL: return "null pointer";
    case MOE_ERR_SHAPE: return "unsupported shape";
    case MOE_ERR_ALIGN: return "misaligned pointer";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_UNSUPPORTED: return "unsupported request";
  }
  return "unknown status";
}

extern "C" const char* moe_last_error(void) { return g_last_error; }

// ------------------------------------------ allocation-free layer variant --
// moe_layer_noalloc: the whole layer with the intermediate kept in a fixed
// array that belongs to this library instead of a caller-provided buffer, for
// callers that cannot allocate device memory themselves. The array lives for
// as long as the library is loaded, on every GPU that uses it.

static __device__ __align__(256) uint16_t g_noalloc_intermediate[MOE_NOALLOC_MAX_INTERMEDIATE];

namespace {

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mutex;
uint16_t* g_noalloc_ptr[kNoAllocMaxDevices] = {};

// Device address of the fixed intermediate array on the current device. Host
// code must not pass the array's name to a kernel (on the host it only stands
// for the symbol), so the address is looked up once per device, with that
// device current, and cached.
moe_status noalloc_intermediate(uint16_t** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    set_error("moe_layer_noalloc: cudaGetDevice", e);
    return MOE_ERR_CUDA;
  }
  if (dev < 0 || dev >= kNoAllocMaxDevices) {
    set_error_msg("moe_layer_noalloc: device index beyond the supported 64 devices");
    return MOE_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_intermediate);
    if (e != cudaSuccess) {
      set_error("moe_layer_noalloc: cudaGetSymbolAddress", e);
      return MOE_ERR_CUDA;
    }
    g_noalloc_ptr[dev] = static_cast<uint16_t*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return MOE_OK;
}

}  // namespace

extern "C" moe_status moe_layer_noalloc(const moe_shape* shape, const moe_weights* w,
                                        const uint16_t* x, const int32_t* ids, const float* wts,
                                        int32_t B, float* y, int32_t* err_flag, void* stream) {
  moe_status rc = check_shape(shape, B);
  if (rc != MOE_OK) return rc;
  if ((rc = check_weights(w, true, true)) != MOE_OK) return rc;
  if (B == 0) return MOE_OK;
  if (!x || !ids || !wts || !y) return MOE_ERR_NULL;
  const size_t need = (size_t)B * (size_t)shape->top_k * (size_t)shape->I;
  if (need > (size_t)MOE_NOALLOC_MAX_INTERMEDIATE) {
    snprintf(g_last_error, sizeof(g_last_error),
             "moe_layer_noalloc: B*top_k*I = %zu BF16 values exceeds the fixed intermediate "
             "capacity of %zu; use moe_layer with a caller-provided buffer",
             need, (size_t)MOE_NOALLOC_MAX_INTERMEDIATE);
    return MOE_ERR_SHAPE;
  }
  uint16_t* h = nullptr;
  if ((rc = noalloc_intermediate(&h)) != MOE_OK) return rc;
  // every intermediate element is written by moe_gate_up (0 for an invalid
  // id) before moe_down reads it on the same stream: nothing needs clearing
  rc = gate_up_impl(shape, w, x, ids, B, h, err_flag, (cudaStream_t)stream);
  if (rc != MOE_OK) return rc;
  return down_impl(shape, w, h, ids, wts, B, y, err_flag, (cudaStream_t)stream, true);
}
