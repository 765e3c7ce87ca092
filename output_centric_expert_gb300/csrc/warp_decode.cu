// GB300 (sm_103a) kernels and C-ABI launchers of the output-centric
// ("warp decode") MoE decode layer.
//
// Method: "Better MoE model inference with warp decode" (Key claims
// [§Reorganized parallelism], [§How the two kernels work], [§Warp Independence];
// Method) and the sd114.wiki "Warp Decode" page (section
// 技术原理：两个 Kernel 搞定一切): every warp owns one output scalar, streams the
// weight rows it needs from global memory into a private FP32 accumulator, and
// finishes with a __shfl_xor_sync butterfly -- no shared memory, no barriers,
// no cross-warp communication.
//
// GB300 design:
//  * Each lane owns 16-byte chunks (16 E4M3 codes) of the rows, chunk c of a
//    warp's stream at lane c % 32, so every warp-wide load instruction reads
//    512 contiguous bytes. All of a round's loads are issued before any of
//    them is consumed, to keep bytes in flight (HBM3e latency x bandwidth).
//  * Weights are read with ld.global.nc + L1::no_allocate (streamed once per
//    warp; reuse across tokens happens in the 126 MB L2); activations use the
//    default cached path (the 8 warps of a CTA share them through L1).
//  * Grid order puts the neuron/output block on the slow axis and the
//    (token, slot) on the fast axis, so tokens routed to the same expert read
//    the same rows close together in time and the re-reads hit L2.
//  * MXFP8 decode: each E8M0 scale is applied once per 16-element partial sum
//    (an exact power-of-two scaling); E4M3 codes are converted with the
//    hardware e4m3x2 -> f16x2 conversion, which is exact.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>

#include "warp_decode.h"

namespace {

constexpr int kWarpsPerCta = 8;  // 8 warps per CTA, as the pages give for moe_gate_up
constexpr int kThreads = kWarpsPerCta * 32;
constexpr int kRound = 4;  // 16-byte chunks per lane per load round

// ---------------------------------------------------------------- loads ----

__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
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

// Two E4M3 codes (low byte = first element) -> two FP32 values, exact.
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint32_t two_codes) {
  uint32_t h2;
  const unsigned short in = (unsigned short)two_codes;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
  return __half22float2(*reinterpret_cast<const __half2*>(&h2));
}

// BF16 pair (low half = first element) -> FP32, exact widening.
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// 16 activations (two 16-byte chunks of BF16) -> FP32 registers.
__device__ __forceinline__ void widen16(const uint4& a, const uint4& b, float (&f)[16]) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    f[2 * i] = bf16_lo(w[i]);
    f[2 * i + 1] = bf16_hi(w[i]);
  }
}

// sum_i f[i] * e4m3(code_i) over one 16-byte chunk of codes.
__device__ __forceinline__ float dot16(const uint4& codes, const float (&f)[16]) {
  const uint32_t w[4] = {codes.x, codes.y, codes.z, codes.w};
  float acc = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 lo = e4m3x2_to_f32x2(w[i]);
    const float2 hi = e4m3x2_to_f32x2(w[i] >> 16);
    acc = fmaf(f[4 * i + 0], lo.x, acc);
    acc = fmaf(f[4 * i + 1], lo.y, acc);
    acc = fmaf(f[4 * i + 2], hi.x, acc);
    acc = fmaf(f[4 * i + 3], hi.y, acc);
  }
  return acc;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, m);
  return v;
}

__device__ __forceinline__ void flag_invalid(int32_t* err) {
  if (err) atomicOr(err, 1);
}

// ------------------------------------------------------------ moe_gate_up --
// grid = (B*top_k pairs, ceil(I / 8)); block = 8 warps; warp w of block
// (p, nb) computes neuron n = 8*nb + w of pair p = t*top_k + j.
__global__ void __launch_bounds__(kThreads)
    moe_gate_up_kernel(const uint8_t* __restrict__ gu_codes,
                       const uint8_t* __restrict__ gu_scales,
                       const uint16_t* __restrict__ x, const int32_t* __restrict__ ids,
                       uint16_t* __restrict__ h, int32_t* __restrict__ err, int H, int I,
                       int E, int top_k) {
  const int lane = threadIdx.x & 31;
  const int p = blockIdx.x;
  const int n = blockIdx.y * kWarpsPerCta + (threadIdx.x >> 5);
  if (n >= I) return;
  const int t = p / top_k;
  const int e = __ldg(ids + p);
  if (e < 0 || e >= E) {
    if (lane == 0) {
      h[(size_t)p * I + n] = 0;
      flag_invalid(err);
    }
    return;
  }
  const int chunks = H >> 4;   // 16-byte chunks per row
  const int blocks = H >> 5;   // scales per row
  const uint8_t* grow = gu_codes + ((size_t)e * I + n) * 2 * (size_t)H;  // up row at +H
  const uint8_t* srow = gu_scales + ((size_t)e * I + n) * 2 * (size_t)blocks;
  const uint16_t* xrow = x + (size_t)t * H;

  float g = 0.0f, u = 0.0f;
  for (int c0 = 0; c0 < chunks; c0 += 32 * kRound) {
    uint4 gw[kRound], uw[kRound], xa[kRound], xb[kRound];
    uint32_t gs[kRound], us[kRound];
#pragma unroll
    for (int q = 0; q < kRound; ++q) {
      const int c = c0 + q * 32 + lane;
      if (c < chunks) {
        gw[q] = ld_stream16(grow + (size_t)c * 16);
        uw[q] = ld_stream16(grow + H + (size_t)c * 16);
        xa[q] = ld_cached16(xrow + c * 16);
        xb[q] = ld_cached16(xrow + c * 16 + 8);
        gs[q] = __ldg(srow + (c >> 1));
        us[q] = __ldg(srow + blocks + (c >> 1));
      }
    }
#pragma unroll
    for (int q = 0; q < kRound; ++q) {
      const int c = c0 + q * 32 + lane;
      if (c < chunks) {
        float xf[16];
        widen16(xa[q], xb[q], xf);
        g = fmaf(dot16(gw[q], xf), e8m0_to_f32(gs[q]), g);
        u = fmaf(dot16(uw[q], xf), e8m0_to_f32(us[q]), u);
      }
    }
  }
  g = warp_sum(g);
  u = warp_sum(u);
  if (lane == 0) {
    const float s = g / (1.0f + expf(-g));
    const __nv_bfloat16 hv = __float2bfloat16_rn(s * u);
    h[(size_t)p * I + n] = *reinterpret_cast<const uint16_t*>(&hv);
  }
}

// --------------------------------------------------------------- moe_down --
// grid = (B tokens, ceil(H / 8)); block = 8 warps; warp w of block (t, ob)
// computes output o = 8*ob + w of token t. The top_k down rows form one flat
// stream of top_k * I/16 chunks spread over the lanes; every chunk adds
// (partial dot) * scale * routing weight into the lane's single accumulator.
__global__ void __launch_bounds__(kThreads)
    moe_down_kernel(const uint8_t* __restrict__ d_codes, const uint8_t* __restrict__ d_scales,
                    const uint16_t* __restrict__ h, const int32_t* __restrict__ ids,
                    const float* __restrict__ wts, float* __restrict__ y,
                    int32_t* __restrict__ err, int H, int I, int E, int top_k) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x;
  const int o = blockIdx.y * kWarpsPerCta + (threadIdx.x >> 5);
  if (o >= H) return;
  const int chunks = I >> 4;  // per down row
  const int blocks = I >> 5;
  const int total = top_k * chunks;
  // (slot, chunk-in-row) of this lane's first chunk; advanced by 32 per step
  int j = lane / chunks;
  int r = lane - j * chunks;
  bool bad = false;

  float acc = 0.0f;
  for (int f0 = 0; f0 < total; f0 += 32 * kRound) {
    uint4 cw[kRound], ha[kRound], hb[kRound];
    uint32_t sc[kRound];
    float wj[kRound];
    bool live[kRound];
#pragma unroll
    for (int q = 0; q < kRound; ++q) {
      const int f = f0 + q * 32 + lane;
      live[q] = false;
      if (f < total) {
        const int slot = t * top_k + j;
        const int e = __ldg(ids + slot);
        if (e >= 0 && e < E) {
          const size_t row = (size_t)e * H + o;
          cw[q] = ld_stream16(d_codes + row * I + (size_t)r * 16);
          sc[q] = __ldg(d_scales + row * blocks + (r >> 1));
          ha[q] = ld_cached16(h + (size_t)slot * I + r * 16);
          hb[q] = ld_cached16(h + (size_t)slot * I + r * 16 + 8);
          wj[q] = __ldg(wts + slot);
          live[q] = true;
        } else {
          bad = true;
        }
        r += 32;
        while (r >= chunks) {
          r -= chunks;
          ++j;
        }
      }
    }
#pragma unroll
    for (int q = 0; q < kRound; ++q) {
      if (live[q]) {
        float hf[16];
        widen16(ha[q], hb[q], hf);
        acc = fmaf(dot16(cw[q], hf), e8m0_to_f32(sc[q]) * wj[q], acc);
      }
    }
  }
  acc = warp_sum(acc);
  if (bad) flag_invalid(err);
  if (lane == 0) y[(size_t)t * H + o] = acc;
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
  if ((gate_up && !aligned(w->gu_codes, 16)) || (down && !aligned(w->d_codes, 16))) {
    set_error_msg("alignment: weight codes must be 16-byte aligned");
    return MOE_ERR_ALIGN;
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

moe_status gate_up_impl(const moe_shape* s, const moe_weights* w, const uint16_t* x,
                        const int32_t* ids, int32_t B, uint16_t* h, int32_t* err,
                        cudaStream_t st) {
  moe_status rc = check_shape(s, B);
  if (rc != MOE_OK) return rc;
  if ((rc = check_weights(w, true, false)) != MOE_OK) return rc;
  if (B == 0) return MOE_OK;
  if (!x || !ids || !h) return MOE_ERR_NULL;
  if (!aligned(x, 16) || !aligned(h, 16) || !aligned(ids, 4) || !aligned(err, 4)) {
    set_error_msg("alignment: x and h need 16 bytes, ids and err_flag 4");
    return MOE_ERR_ALIGN;
  }
  const dim3 grid((unsigned)(B * s->top_k), (unsigned)((s->I + kWarpsPerCta - 1) / kWarpsPerCta));
  moe_gate_up_kernel<<<grid, kThreads, 0, st>>>(w->gu_codes, w->gu_scales, x, ids, h, err, s->H,
                                                s->I, s->E, s->top_k);
  return launch_status("moe_gate_up launch");
}

moe_status down_impl(const moe_shape* s, const moe_weights* w, const uint16_t* h,
                     const int32_t* ids, const float* wts, int32_t B, float* y, int32_t* err,
                     cudaStream_t st) {
  moe_status rc = check_shape(s, B);
  if (rc != MOE_OK) return rc;
  if ((rc = check_weights(w, false, true)) != MOE_OK) return rc;
  if (B == 0) return MOE_OK;
  if (!h || !ids || !wts || !y) return MOE_ERR_NULL;
  if (!aligned(h, 16) || !aligned(ids, 4) || !aligned(wts, 4) || !aligned(y, 4) ||
      !aligned(err, 4)) {
    set_error_msg("alignment: h needs 16 bytes, ids/wts/y/err_flag 4");
    return MOE_ERR_ALIGN;
  }
  if ((unsigned)B > 0x7FFFFFFFu) return MOE_ERR_SHAPE;
  const dim3 grid((unsigned)B, (unsigned)((s->H + kWarpsPerCta - 1) / kWarpsPerCta));
  moe_down_kernel<<<grid, kThreads, 0, st>>>(w->d_codes, w->d_scales, h, ids, wts, y, err, s->H,
                                             s->I, s->E, s->top_k);
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
  return down_impl(shape, w, h, ids, wts, B, y, err_flag, (cudaStream_t)stream);
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
  return down_impl(shape, w, h_scratch, ids, wts, B, y, err_flag, (cudaStream_t)stream);
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
