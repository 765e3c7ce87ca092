// moe_gate_up, expert-grouped form: one warp per (expert, 8 intermediate
// neurons), serving every (token, slot) pair routed to that expert.
//
// Each warp still owns its outputs h[t, j, n] outright and writes each one
// once, as in "Better MoE model inference with warp decode" [§How the two
// kernels work] and the sd114.wiki "Warp Decode" page (技术原理): no buffer is
// padded, no activation is gathered into a per-expert copy in global memory,
// and nothing is scattered or combined afterwards. What changes is how the
// weights are consumed: the per-token kernel decodes and multiplies every
// MXFP8 weight once per (token, slot) that uses it, which leaves it limited
// by instruction issue once many pairs share an expert (large batches,
// skewed routing). Here each weight is decoded once per pass and multiplied
// on the tensor cores:
//
//   mma.sync m16n8k16, f16 x f16 -> FP32. MMA rows 0-7 are the gate rows of
//   the warp's 8 neurons, rows 8-15 their up rows, so a lane's accumulator
//   fragment holds gate and up of one neuron for two pairs and the SwiGLU
//   epilogue needs no exchange between lanes. The 8 columns are 8 of the
//   expert's routed pairs (two column tiles per pass where shared memory
//   allows, and several passes over the rows when more pairs are routed).
//
// Reduction order. The contraction over H runs block by block: within one
// 32-element MXFP8 block the two MMAs sum the exact f16 x E4M3 products in
// FP32 (the tensor core's own order), the block sum is multiplied by the
// block's E8M0 scale and added to an FP32 accumulator. The k axis inside a
// block is permuted identically for both operands: a quad of lanes loads 64
// contiguous codes (two blocks, 16 codes per lane), the lanes q and q^2 swap
// their upper 8 codes, and then lane q holds 8 codes of each block, at
// element offset 16(q&1) + 8(q>>1) of the even block and 16(q&1) +
// 8(1-(q>>1)) of the odd one; its activation reads use the same offsets. A
// column's result depends only on its own pair, never on the other columns,
// so a token's intermediate does not depend on the rest of the batch.
//
// Work. One CTA per (expert, 64-neuron tile); the CTA ranks the pairs routed
// to its expert in pair order (CTAs of experts without pairs exit at once)
// and stages their tokens' activations in shared memory as the same
// f16 x 2^sigma copy of the BF16 row as the per-token kernel (sigma per
// token). Codes stream through registers, double-buffered 8 blocks deep.
//
// Loads. A warp load reads 64 contiguous bytes of each of 8 rows. With 8
// bytes per lane (32 bytes per row) the L1 data pipe was the busiest unit
// (about 60 % of peak against 47 % for DRAM, ncu, Qwen-3-30B-A3B shape at 32
// tokens); 16 bytes per lane and the swap cut the kernel's time there from
// 95.5 to 83.7 us with bit-identical results. Measured on GB300 it is faster
// than the per-token kernel from about 36 tokens (Qwen-3-30B-A3B shape) or
// 17 tokens (Qwen-3-235B-A22B shape) under uniform routing, and at 32 tokens
// under skewed routing.
#include "wd_device.cuh"
#include "wd_gate_up_grouped.h"

namespace wd {
namespace {

constexpr int kGrpNeuronsPerWarp = 8;                            // MMA rows: 8 gate + 8 up
constexpr int kGrpNeurons = kWarpsPerCta * kGrpNeuronsPerWarp;  // 64 neurons per CTA
constexpr int kGrpCols = 8;                                      // pairs per MMA column tile

// Shared-memory row of one staged token: H f16 plus 64 bytes, which puts
// consecutive tokens 16 banks apart so the 16-byte column reads of a quarter
// warp (two tokens x four lanes) hit distinct banks.
__host__ __device__ constexpr int grp_row_bytes(int H) { return 2 * H + 64; }

// UNR: 32-element blocks per loop step (a multiple of 8: one 64-bit load of
// scales per row per 8 blocks). NCH: column tiles of 8 pairs held at once.
template <int UNR>
struct GrpBuf {
  uint4 g[UNR / 2], u[UNR / 2];    // this lane's 16 codes of each block pair, gate and up
  uint2 sg[UNR / 8], su[UNR / 8];  // scales, 8 blocks per pair of words
};

template <int UNR, int NCH>
__global__ void __launch_bounds__(kThreads, 2)
    moe_gate_up_grouped_kernel(const uint8_t* __restrict__ gu_codes,
                               const uint8_t* __restrict__ gu_scales,
                               const uint16_t* __restrict__ x, const int32_t* __restrict__ ids,
                               uint16_t* __restrict__ h, int32_t* __restrict__ err, int H, int I,
                               int E, int top_k, int B) {
  static_assert(UNR % 8 == 0, "UNR: multiple of 8");
  constexpr int kT = NCH * kGrpCols;  // pairs staged per pass
  extern __shared__ uint4 xs4[];      // [kT] rows of grp_row_bytes(H)
  __shared__ int s_pair[kT];          // pair index t*top_k + j of each staged column
  __shared__ int s_sig[kT];           // its activation scale exponent
  __shared__ int s_wcnt[kWarpsPerCta];

  const int tiles = I / kGrpNeurons;
  const int e = blockIdx.x / tiles;
  const int tile = blockIdx.x - e * tiles;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;  // MMA group (neuron) and lane in the quad
  const int n = tile * kGrpNeurons + warp * kGrpNeuronsPerWarp + g;
  const int P = B * top_k;
  const int nblk = H >> 5;
  const int RS = grp_row_bytes(H);
  uint8_t* xs = reinterpret_cast<uint8_t*>(xs4);

  launch_dependents();

  // A pair whose id is outside [0, E) belongs to no expert: the CTAs of
  // expert 0 write its zeros over their neurons and raise the flag.
  if (e == 0) {
    for (int p = threadIdx.x; p < P; p += kThreads) {
      const int id = __ldg(ids + p);
      if (id < 0 || id >= E) {
        flag_invalid(err);
        uint4* o = reinterpret_cast<uint4*>(h + (size_t)p * I + tile * kGrpNeurons);
#pragma unroll
        for (int i = 0; i < kGrpNeurons / 8; ++i) o[i] = make_uint4(0, 0, 0, 0);
      }
    }
  }

  const uint8_t* grow = gu_codes + ((size_t)e * I + n) * 2 * H + q * 16;  // gate row, lane's 16 B
  const uint8_t* urow = grow + H;
  const uint8_t* gsc = gu_scales + ((size_t)e * I + n) * 2 * nblk;
  const uint8_t* usc = gsc + nblk;
  const uint8_t* xl = xs + g * RS;  // column g of tile 0

  auto load = [&](int it, GrpBuf<UNR>& U) {
    const int b0 = it * UNR;
#pragma unroll
    for (int i = 0; i < UNR / 2; ++i) {
      U.g[i] = ld_codes16(grow + (size_t)(b0 + 2 * i) * 32);
      U.u[i] = ld_codes16(urow + (size_t)(b0 + 2 * i) * 32);
    }
#pragma unroll
    for (int i = 0; i < UNR / 8; ++i) {
      U.sg[i] = ld_scales8(gsc + b0 + 8 * i);
      U.su[i] = ld_scales8(usc + b0 + 8 * i);
    }
  };
  // element offset of this lane's 8 codes in an even and an odd block
  const int off_even = 16 * (q & 1) + 8 * (q >> 1);
  const int off_odd = 16 * (q & 1) + 8 * (1 - (q >> 1));
  const bool low = q < 2;

  for (int lo = 0;; lo += kT) {
    // Rank the pairs routed to expert e in pair order; keep ranks [lo, lo+kT).
    int n_e = 0;
    for (int p0 = 0; p0 < P; p0 += kThreads) {
      const int p = p0 + threadIdx.x;
      const bool mine = p < P && __ldg(ids + p) == e;
      const unsigned bal = __ballot_sync(0xFFFFFFFFu, mine);
      if (lane == 0) s_wcnt[warp] = __popc(bal);
      __syncthreads();
      int rank = n_e + __popc(bal & ((1u << lane) - 1u));
#pragma unroll
      for (int w = 0; w < kWarpsPerCta; ++w) {
        const int c = s_wcnt[w];
        rank += (w < warp) ? c : 0;
        n_e += c;
      }
      if (mine && rank >= lo && rank < lo + kT) s_pair[rank - lo] = p;
      __syncthreads();
    }
    if (lo >= n_e) break;  // the same decision in every thread
    const int cols = min(kT, n_e - lo);
    const int nch = (cols + kGrpCols - 1) / kGrpCols;

    // the first codes are requested before the activations are staged
    GrpBuf<UNR> U0, U1;
    load(0, U0);

    // Stage the columns: warp c converts pair c's token row to f16 x 2^sigma.
    for (int c = warp; c < cols; c += kWarpsPerCta) {
      const int t = s_pair[c] / top_k;
      const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H);
      float m = 0.0f;
      for (int i = lane; i < (H >> 3); i += 32) m = fmaxf(m, absmax8(ld_cached16(src + i)));
      const int sigma = pow2_shift_for(warp_max(m));
      const float up = exp2i(sigma);
      uint4* dst = reinterpret_cast<uint4*>(xs + (size_t)c * RS);
      for (int i = lane; i < (H >> 3); i += 32) dst[i] = to_f16x8(ld_cached16(src + i), up);
      if (lane == 0) s_sig[c] = sigma;
    }
    __syncthreads();

    float accg[NCH][2], accu[NCH][2];
#pragma unroll
    for (int c = 0; c < NCH; ++c) accg[c][0] = accg[c][1] = accu[c][0] = accu[c][1] = 0.0f;
    const float zero[4] = {0.0f, 0.0f, 0.0f, 0.0f};

    auto compute = [&](int it, const GrpBuf<UNR>& U) {
#pragma unroll
      for (int i2 = 0; i2 < UNR / 2; ++i2) {
        // swap upper halves with lane q^2: each lane then holds 8 codes of both blocks
        const uint32_t rg2 = __shfl_xor_sync(0xFFFFFFFFu, U.g[i2].z, 2);
        const uint32_t rg3 = __shfl_xor_sync(0xFFFFFFFFu, U.g[i2].w, 2);
        const uint32_t ru2 = __shfl_xor_sync(0xFFFFFFFFu, U.u[i2].z, 2);
        const uint32_t ru3 = __shfl_xor_sync(0xFFFFFFFFu, U.u[i2].w, 2);
        const uint2 cgb[2] = {low ? make_uint2(U.g[i2].x, U.g[i2].y) : make_uint2(rg2, rg3),
                              low ? make_uint2(rg2, rg3) : make_uint2(U.g[i2].x, U.g[i2].y)};
        const uint2 cub[2] = {low ? make_uint2(U.u[i2].x, U.u[i2].y) : make_uint2(ru2, ru3),
                              low ? make_uint2(ru2, ru3) : make_uint2(U.u[i2].x, U.u[i2].y)};
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
          const int i = 2 * i2 + hb;
          const int b = it * UNR + i;
          uint32_t a0[4], a1[4];
          e4m3x4_to_f16x4(cgb[hb].x, a0[0], a0[2]);
          e4m3x4_to_f16x4(cub[hb].x, a0[1], a0[3]);
          e4m3x4_to_f16x4(cgb[hb].y, a1[0], a1[2]);
          e4m3x4_to_f16x4(cub[hb].y, a1[1], a1[3]);
          const uint32_t swd = (i % 8) < 4 ? U.sg[i / 8].x : U.sg[i / 8].y;
          const uint32_t uwd = (i % 8) < 4 ? U.su[i / 8].x : U.su[i / 8].y;
          float sg, su;
          e8m0x2_to_f32(swd >> (8 * (i % 4)), uwd >> (8 * (i % 4)), sg, su);
          const int off = hb ? off_odd : off_even;
#pragma unroll
          for (int c = 0; c < NCH; ++c) {
            if (c < nch) {
              const uint4 xv = *reinterpret_cast<const uint4*>(
                  xl + (size_t)c * kGrpCols * RS + b * 64 + 2 * off);
              float d[4];
              mma_16816(d, a0, xv.x, xv.y, zero);
              mma_16816(d, a1, xv.z, xv.w, d);
              accg[c][0] = fmaf(d[0], sg, accg[c][0]);
              accg[c][1] = fmaf(d[1], sg, accg[c][1]);
              accu[c][0] = fmaf(d[2], su, accu[c][0]);
              accu[c][1] = fmaf(d[3], su, accu[c][1]);
            }
          }
        }
      }
    };

    const int nit = nblk / UNR;
    for (int it = 0; it < nit; it += 2) {
      if (it + 1 < nit) load(it + 1, U1);
      compute(it, U0);
      if (it + 1 < nit) {
        if (it + 2 < nit) load(it + 2, U0);
        compute(it + 1, U1);
      }
    }

    // Epilogue: lane (g, q) holds gate and up of neuron n for columns 2q, 2q+1.
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int li = c * kGrpCols + 2 * q + k;
        if (li < cols) {
          const float unscale = exp2i(-s_sig[li]);
          const float gv = accg[c][k] * unscale, uv = accu[c][k] * unscale;
          const float sl = gv / (1.0f + expf(-gv));
          const __nv_bfloat16 hv = __float2bfloat16_rn(sl * uv);
          h[(size_t)s_pair[li] * I + n] = *reinterpret_cast<const uint16_t*>(&hv);
        }
      }
    }
    __syncthreads();  // the next pass restages the columns
  }
}

template <int UNR, int NCH>
moe_status launch_grouped(const moe_shape* s, const moe_weights* w, const uint16_t* x,
                          const int32_t* ids, int32_t B, uint16_t* h, int32_t* err,
                          cudaStream_t st) {
  const size_t smem = (size_t)NCH * kGrpCols * grp_row_bytes(s->H);
  moe_status rc = allow_smem(moe_gate_up_grouped_kernel<UNR, NCH>, smem);
  if (rc != MOE_OK) return rc;
  const unsigned grid = (unsigned)(s->E * (s->I / kGrpNeurons));
  moe_gate_up_grouped_kernel<UNR, NCH><<<grid, kThreads, smem, st>>>(
      w->gu_codes, w->gu_scales, x, ids, h, err, s->H, s->I, s->E, s->top_k, B);
  return MOE_OK;
}

constexpr int kGrpUnroll = 8;

}  // namespace

bool gate_up_grouped_supported(const moe_shape* s, const moe_weights* w) {
  return s->H % (32 * kGrpUnroll) == 0 && s->I % kGrpNeurons == 0 &&
         (w == nullptr || aligned(w->gu_scales, 8)) &&
         (size_t)kGrpCols * grp_row_bytes(s->H) <= kMaxDynSmem &&
         (int64_t)s->E * (s->I / kGrpNeurons) <= 0x7FFFFFFF;
}

moe_status launch_gate_up_grouped(const moe_shape* s, const moe_weights* w, const uint16_t* x,
                                  const int32_t* ids, int32_t B, uint16_t* h, int32_t* err,
                                  cudaStream_t st) {
  // two column tiles per pass when 16 staged rows still leave room for two
  // CTAs per SM
  if ((size_t)2 * kGrpCols * grp_row_bytes(s->H) <= 100 * 1024)
    return launch_grouped<kGrpUnroll, 2>(s, w, x, ids, B, h, err, st);
  return launch_grouped<kGrpUnroll, 1>(s, w, x, ids, B, h, err, st);
}

}  // namespace wd
