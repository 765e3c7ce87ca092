// Device code shared by the kernels of the output-centric ("warp decode")
// MoE decode layer for GB300 (sm_103a), and the host helpers their
// launchers share.
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
//  * Latency is hidden by occupancy. moe_gate_up stays at 80 registers, so 3
//    CTAs (24 warps) fit on an SM; its warps loop over several routed slots of
//    one token. moe_down warps own several outputs that share one read of the
//    intermediate from shared memory. They use 80 registers with at most 4
//    rows in flight per lane, and 128 registers (2 CTAs per SM) when a lane
//    holds 8 rows' codes: 8 outputs, or fewer outputs with several units at
//    once on small batches. (Holding a second unit of codes to prefetch it,
//    staging codes through a cp.async or bulk-copy ring in shared memory, and
//    refilling registers row by row all measured slower on this part.)
//  * Row strides. The kernels are also compiled with the row length as a
//    constant for the hidden and intermediate sizes of the target layers, so
//    strides and offsets are load immediates (wd_gate_up_fixed.cu, wd_down.cu).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>

#include "warp_decode.h"

namespace wd {

constexpr int kWarpsPerCta = 8;  // 8 warps per CTA, as the pages give for moe_gate_up
constexpr int kThreads = kWarpsPerCta * 32;
constexpr int kSegBlocksPerLane = 2;               // gate/up: 32-element blocks per lane per unit
constexpr int kSegBlocks = 32 * kSegBlocksPerLane;  // blocks of one row per unit (2048 elements)
constexpr int kMinCtasPerSm = 8;                    // CTAs per SM that fill the GPU several times

constexpr int kRouteMaxE = 256;

struct RouteArgs {
  const float* logits;  // [B][E], or nullptr: the ids/wts arrays are the routing
  bool dependent;       // launched as a programmatic dependent of the router kernel
                        // that writes the ids (the kernel waits before reading them)
};

constexpr RouteArgs kNoRoute = {nullptr, false};

// ------------------------------------------------------ host helpers (shared) --
// Defined with the C-ABI entry points; one error message per calling thread.
void set_error(const char* what, cudaError_t e);
void set_error_msg(const char* msg);

inline bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p % a) == 0; }

// Number of SMs of the current device (looked up once per device; 152 on a
// GB300). Only the launch heuristics use it: grids stay correct for any value.
int sm_count();

constexpr size_t kMaxDynSmem = 227 * 1024;

// Opt a kernel into more than the default 48 KB of dynamic shared memory.
template <typename K>
inline moe_status allow_smem(K kernel, size_t bytes) {
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

// Launchers of the two kernels (wd_gate_up.cu, wd_down.cu); the arguments
// have been validated by the C-ABI entry points. They return MOE_OK or an
// error status, and check nothing that the entry points check.
moe_status launch_gate_up_kernels(const moe_shape* s, const moe_weights* w, const uint16_t* x,
                                  const int32_t* ids, int32_t B, uint16_t* h, int32_t* err,
                                  cudaStream_t st, RouteArgs route);
// moe_gate_up with a kernel compiled for the shape's H, if there is one:
// returns false (launching nothing) otherwise. spw: routed slots per warp;
// ctas_per_sm: 3, or 4 (64 registers; 2 or 4 slots per warp).
bool launch_gate_up_fixed_h(const moe_shape* s, const moe_weights* w, const uint16_t* x,
                            const int32_t* ids, int32_t B, uint16_t* h, int32_t* err,
                            cudaStream_t st, RouteArgs route, int spw, int ctas_per_sm,
                            moe_status* rc);
// dependent = true launches moe_down as a programmatic dependent of the kernel
// before it on the stream (used by the layer entry points, where that kernel
// is moe_gate_up and only h is produced by it).
moe_status launch_down_kernels(const moe_shape* s, const moe_weights* w, const uint16_t* h,
                               const int32_t* ids, const float* wts, int32_t B, float* y,
                               int32_t* err, cudaStream_t st, bool dependent,
                               const float* logits);

namespace {  // device code: one copy per translation unit

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

// d = a * b + c for one m16n8k16 tile: f16 operands, FP32 accumulate.
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1, const float (&c)[4]) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%11,%12,%13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]),
        "f"(c[2]), "f"(c[3]));
}

// 16 codes (half of one of two adjacent 32-element blocks), not allocated in
// L1. A warp's load covers 64 bytes of each of 8 rows and its next three loads
// the rest of the same 256 bytes, so the L2 fetches 256-byte segments
// (grouped gate/up alone: Qwen-3-30B-A3B 32 tokens 68.7 -> 68.4 us,
// Qwen-3-235B-A22B 32 tokens 237.3 -> 235.4, Mixtral-shaped 16 tokens 159.5 ->
// 158.4; 128-byte segments: no change).
__device__ __forceinline__ uint4 ld_codes16(const uint8_t* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}
// The E8M0 scales of 8 consecutive blocks of one row.
__device__ __forceinline__ uint2 ld_scales8(const uint8_t* p) {
  uint2 r;
  asm("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
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

// Two E8M0 scale codes (bits 0..7 of lo and of hi) -> 2^(s-127) as FP32 each,
// through the hardware E8M0 -> BF16x2 conversion: BF16 has E8M0's 8-bit
// exponent, so the conversion is exact (code 0 gives the subnormal 2^-127,
// code 255 a NaN; checked on all 256 codes on GB300), and a BF16 widens to
// FP32 by a shift. One conversion replaces two five-instruction decodes.
__device__ __forceinline__ void e8m0x2_to_f32(uint32_t lo, uint32_t hi, float& a, float& b) {
  const uint32_t two = __byte_perm(lo, hi, 0x0040);  // lo byte 0, hi byte 0
  uint32_t r;
  asm("{.reg .b16 p, q;\n\t"
      "mov.b32 {p, q}, %1;\n\t"
      "cvt.rn.bf16x2.ue8m0x2 %0, p;\n\t}"
      : "=r"(r)
      : "r"(two));
  a = __uint_as_float(r << 16);
  b = __uint_as_float(r & 0xFFFF0000u);
}

// The four E8M0 codes of w (byte i -> f[i]), as above.
__device__ __forceinline__ void e8m0x4_to_f32(uint32_t w, float (&f)[4]) {
  uint32_t r0, r1;
  asm("{.reg .b16 a, b;\n\t"
      "mov.b32 {a, b}, %2;\n\t"
      "cvt.rn.bf16x2.ue8m0x2 %0, a;\n\t"
      "cvt.rn.bf16x2.ue8m0x2 %1, b;\n\t}"
      : "=r"(r0), "=r"(r1)
      : "r"(w));
  f[0] = __uint_as_float(r0 << 16);
  f[1] = __uint_as_float(r0 & 0xFFFF0000u);
  f[2] = __uint_as_float(r1 << 16);
  f[3] = __uint_as_float(r1 & 0xFFFF0000u);
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
// Returns sigma. Must be called by all threads of the CTA. HOLD: when every
// thread's share is at most kHeld pieces, keep them in registers between the
// max pass and the conversion instead of reading them again (used by
// moe_down: Q30 B=32 44.0 -> 43.0 us; in moe_gate_up it slowed the
// 235B-shaped layer).
constexpr int kHeld = 4;
template <bool HOLD = false>
__device__ int stage_activations(const uint16_t* __restrict__ src, int rows, int len,
                                 uint4* dst, float* red) {
  const int pieces_per_row = len >> 3;  // 16-byte pieces (8 elements)
  const int pieces = rows * pieces_per_row;
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
  float m = 0.0f;
  if (HOLD && pieces <= kHeld * kThreads) {
    uint4 v[kHeld];
#pragma unroll
    for (int i = 0; i < kHeld; ++i) {
      const int p = threadIdx.x + i * kThreads;
      v[i] = p < pieces ? ld_cached16(s4 + p) : make_uint4(0, 0, 0, 0);
      m = fmaxf(m, absmax8(v[i]));
    }
    m = warp_max(m);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    m = red[0];
#pragma unroll
    for (int i = 1; i < kWarpsPerCta; ++i) m = fmaxf(m, red[i]);
    const int sigma = pow2_shift_for(m);
    const float up = exp2i(sigma);
    const int nblk = len >> 5;
#pragma unroll
    for (int i = 0; i < kHeld; ++i) {
      const int p = threadIdx.x + i * kThreads;
      if (p < pieces) {
        const int r = p / pieces_per_row, q = p - r * pieces_per_row;
        dst[r * pieces_per_row + (q & 3) * nblk + (q >> 2)] = to_f16x8(v[i], up);
      }
    }
    __syncthreads();
    return sigma;
  }
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

}  // namespace
}  // namespace wd
