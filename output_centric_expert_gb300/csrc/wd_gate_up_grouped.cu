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
//   expert's routed pairs (several passes over the rows when more pairs are
//   routed).
//
// Reduction order. The contraction over H runs block by block: within one
// 32-element MXFP8 block the two MMAs sum the exact f16 x E4M3 products in
// FP32 (the tensor core's own order), the block sum is multiplied by the
// block's E8M0 scale and added to an FP32 accumulator; the blocks of the
// lower half of H and those of the upper half go to two accumulators, added
// at the end (lower + upper), however the item is run. The k axis inside a
// block is permuted identically for both operands: a quad of lanes loads 64
// contiguous codes (two blocks, 16 codes per lane), the lanes q and q^2 swap
// their upper 8 codes, and then lane q holds 8 codes of each block, at
// element offset 16(q&1) + 8(q>>1) of the even block and 16(q&1) +
// 8(1-(q>>1)) of the odd one; its activation reads use the same offsets. A
// column's result depends only on its own pair, never on the other columns,
// so a token's intermediate does not depend on the rest of the batch.
//
// Work. A persistent grid of two CTAs per SM. Every CTA lists the batch's
// pairs by expert in pair order and numbers the work items (expert, pass of
// up to 8 pairs, 64-neuron tile) with the items of one (expert, pass)
// consecutive; CTA c takes the c-th contiguous share, counted in half-items
// of 32 neurons where that lowers the largest share. A half-item without its
// partner in the share runs on all 8 warps, each half of H on 4 of them, and
// the two partial sums meet in shared memory: at 4.5 items per CTA (the
// Qwen-3-30B-A3B shape at 32 tokens) the CTAs with 5 whole items left the
// others idle for a fifth of the kernel (74.0 -> 69.0 us; 64 tokens 83.5 ->
// 79.7, skewed 32 tokens 45.6 -> 41.9, Qwen-3-235B-A22B 64 tokens 281.3 ->
// 269.4, Mixtral-shaped 8 tokens 147.0 -> 138.0). For each new (expert,
// pass) the CTA stages its pairs' activations in shared memory as the same
// f16 x 2^sigma copy of the BF16 row as the per-token kernel (sigma per
// token) and keeps them for the pass's following tiles. Codes stream through
// registers, double-buffered 8 blocks deep, and each warp requests the first
// codes of its next item while it computes the last ones of the current item.
// Against one CTA per (expert, tile), which ranked its expert's pairs and
// staged them in every CTA, this measured bit-identical and faster for the
// Qwen-3-30B-A3B shape (64 tokens 97.0 -> 94.2 us, skewed 74.7 -> 59.5 us),
// about 3 % slower for the Qwen-3-235B-A22B shape at 32-64 tokens; a grid of
// four CTAs per SM was slower everywhere (the lists are built per CTA).
//
// Loads. A warp load reads 64 contiguous bytes of each of 8 rows. With 8
// bytes per lane (32 bytes per row) the L1 data pipe was the busiest unit
// (about 60 % of peak against 47 % for DRAM, ncu, Qwen-3-30B-A3B shape at 32
// tokens); 16 bytes per lane and the swap cut the kernel's time there from
// 95.5 to 83.7 us with bit-identical results. Measured on GB300, in the
// layer, it is faster than the per-token kernel from about 25 tokens
// (Qwen-3-30B-A3B shape) or 24 tokens (Qwen-3-235B-A22B shape) under uniform
// routing, and far ahead at 32 skewed tokens.
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
// scales per row per 8 blocks).
template <int UNR>
struct GrpBuf {
  uint4 g[UNR / 2], u[UNR / 2];    // this lane's 16 codes of each block pair, gate and up
  uint2 sg[UNR / 8], su[UNR / 8];  // scales, 8 blocks per pair of words
};

// Byte offsets of the kernel's shared-memory arrays.
struct GrpLayout {
  size_t xs, list, cnt, start, istart, run, wc, total;
};

__host__ __device__ inline GrpLayout grp_layout(int H, int E, int P) {
  GrpLayout L;
  size_t o = 0;
  L.xs = o;      // [kGrpCols] staged activation rows of grp_row_bytes(H)
  o += (size_t)kGrpCols * grp_row_bytes(H);
  L.list = o;    // [P] int: pair indices grouped by expert, in pair order
  o += (size_t)P * 4;
  L.cnt = o;     // [E] int: pairs routed to each expert
  o += (size_t)E * 4;
  L.start = o;   // [E] int: first list entry of each expert
  o += (size_t)E * 4;
  L.istart = o;  // [E + 1] int: first work item of each expert; [E] = the number of items
  o += (size_t)(E + 1) * 4;
  L.run = o;     // [E] int: entries placed so far
  o += (size_t)E * 4;
  L.wc = o;      // [warp][E] int: per-warp counts while placing; afterwards the
                 // upper-half partial sums of a split half-item, [4 warps][32 lanes][4] float
  o += (size_t)(kWarpsPerCta * E > 4 * 32 * 4 ? kWarpsPerCta * E : 4 * 32 * 4) * 4;
  L.total = o;
  return L;
}

// Persistent: a grid of two CTAs per SM. Every CTA lists the batch's pairs by
// expert (in pair order) and numbers the work items (expert, pass of kT pairs,
// 64-neuron tile), items of one (expert, pass) consecutive; CTA c takes the
// c-th contiguous share of the items or half-items. The staged activations of
// a pass serve all of its tiles that fall to the CTA, and each warp requests
// the first codes of its next unit while it computes the last ones of the
// current unit.
template <int UNR>
__global__ void __launch_bounds__(kThreads, 2)
    moe_gate_up_grouped_kernel(const uint8_t* __restrict__ gu_codes,
                               const uint8_t* __restrict__ gu_scales,
                               const uint16_t* __restrict__ x, const int32_t* __restrict__ ids,
                               uint16_t* __restrict__ h, int32_t* __restrict__ err, int H, int I,
                               int E, int top_k, int B) {
  static_assert(UNR % 8 == 0, "UNR: multiple of 8");
  constexpr int kT = kGrpCols;  // pairs staged per pass
  constexpr unsigned kFull = 0xFFFFFFFFu;
  extern __shared__ uint4 dyn4[];
  __shared__ int s_pair[kT];          // pair index t*top_k + j of each staged column
  __shared__ int s_sig[kT];           // its activation scale exponent
  __shared__ int s_wtot[2][kWarpsPerCta];

  const int P = B * top_k;
  const GrpLayout L = grp_layout(H, E, P);
  uint8_t* dsm = reinterpret_cast<uint8_t*>(dyn4);
  uint8_t* xs = dsm + L.xs;
  int* s_list = reinterpret_cast<int*>(dsm + L.list);
  int* s_cnt = reinterpret_cast<int*>(dsm + L.cnt);
  int* s_start = reinterpret_cast<int*>(dsm + L.start);
  int* s_istart = reinterpret_cast<int*>(dsm + L.istart);
  int* s_run = reinterpret_cast<int*>(dsm + L.run);
  int* s_wc = reinterpret_cast<int*>(dsm + L.wc);

  const int tiles = I / kGrpNeurons;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, q = lane & 3;  // MMA group (neuron) and lane in the quad
  const int nblk = H >> 5;
  const int RS = grp_row_bytes(H);

  // ---- pair lists by expert and the work items (the same in every CTA) ----
  for (int i = tid; i < E; i += kThreads) {
    s_cnt[i] = 0;
    s_run[i] = 0;
  }
  for (int i = tid; i < kWarpsPerCta * E; i += kThreads) s_wc[i] = 0;
  wait_prerequisite();  // the ids are complete from here on (a router may write them)
  // moe_down, a dependent of this kernel, reads the ids before its own wait:
  // it is released only now
  launch_dependents();
  __syncthreads();
  for (int p = tid; p < P; p += kThreads) {
    const int id = __ldg(ids + p);
    if (id >= 0 && id < E) atomicAdd(s_cnt + id, 1);
  }
  __syncthreads();
  {  // exclusive scans over the experts (E <= kThreads: one each): list
     // offsets and item offsets (tiles x passes of kT pairs per expert)
    const int c = tid < E ? s_cnt[tid] : 0;
    const int items = tiles * ((c + kT - 1) / kT);
    int ic = c, ii = items;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int a = __shfl_up_sync(kFull, ic, d), b = __shfl_up_sync(kFull, ii, d);
      if (lane >= d) {
        ic += a;
        ii += b;
      }
    }
    if (lane == 31) {
      s_wtot[0][warp] = ic;
      s_wtot[1][warp] = ii;
    }
    __syncthreads();
    int bc = 0, bi = 0;
    for (int w = 0; w < warp; ++w) {
      bc += s_wtot[0][w];
      bi += s_wtot[1][w];
    }
    if (tid < E) {
      s_start[tid] = bc + ic - c;
      s_istart[tid] = bi + ii - items;
    }
    if (tid == kThreads - 1) s_istart[E] = bi + ii;
  }
  __syncthreads();
  // place the pairs in pair order: within a warp by match, across warps by
  // the warps' counts of the same expert, across rounds by the running count
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int c0 = 0; c0 < P; c0 += kThreads) {
    const int p = c0 + tid;
    const int id = p < P ? __ldg(ids + p) : -1;
    const bool valid = id >= 0 && id < E;
    const unsigned m = __match_any_sync(kFull, valid ? id : -1);
    const int lt = __popc(m & lt_mask);
    if (valid && lt == 0) s_wc[warp * E + id] = __popc(m);
    __syncthreads();
    if (valid) {
      int r = s_run[id] + lt;
      for (int w = 0; w < warp; ++w) r += s_wc[w * E + id];
      s_list[s_start[id] + r] = p;
    }
    __syncthreads();
    if (valid && lt == 0) {
      atomicAdd(s_run + id, __popc(m));
      s_wc[warp * E + id] = 0;
    }
    __syncthreads();
  }

  // A pair whose id is outside [0, E) belongs to no expert: its intermediate
  // is 0; CTA c writes the zeros of its share of the I neurons.
  {
    const int per = (I + (int)gridDim.x - 1) / (int)gridDim.x;
    const int n0 = blockIdx.x * per, n1 = min(I, n0 + per);
    for (int p = tid; p < P; p += kThreads) {
      const int id = __ldg(ids + p);
      if (id < 0 || id >= E) {
        if (blockIdx.x == 0) flag_invalid(err);
        for (int nn = n0; nn < n1; ++nn) h[(size_t)p * I + nn] = 0;
      }
    }
  }

  // Work units. A half-item is 32 of an item's 64 neurons, and CTA c takes the
  // c-th contiguous share of the 2 * nitems half-items, so that the shares
  // differ by at most one half-item. Two half-items of one item run as the
  // whole item (warp w: neurons 8w .. 8w+7 over all of H); a half-item whose
  // partner is outside the share runs alone on all 8 warps, warps w and w+4
  // taking neurons 8(w&3) .. of it over the lower and the upper half of H,
  // and the two partial sums are added in shared memory. Every item sums the
  // lower and the upper half of H separately and adds the two at the end,
  // whichever way it runs, so a result does not depend on how the batch fell
  // into shares. (Rows of one 8-block group: whole items only.)
  static_assert(kWarpsPerCta == 8, "a split half-item pairs warps w and w + 4");
  const int nitems = s_istart[E];
  const int nit = nblk / UNR;
  const int half = nit >= 2 ? nit / 2 : nit;  // groups summed into the lower partial
  // shares in half-items where that lowers the largest share (an odd number
  // of half-items at most per CTA); else in whole items, which run no split
  const bool halves =
      nit >= 2 && ((2 * (int64_t)nitems + gridDim.x - 1) / gridDim.x) % 2 == 1;
  const int64_t nunits = halves ? 2 * (int64_t)nitems : (int64_t)nitems;
  const int u0 = (int)(nunits * blockIdx.x / gridDim.x);
  const int u1 = (int)(nunits * (blockIdx.x + 1) / gridDim.x);
  if (u0 >= u1) return;  // the same for every thread of the CTA

  auto is_single = [&](int u) { return halves && ((u & 1) || u + 1 >= u1); };
  auto item_of = [&](int u) { return halves ? (u >> 1) : u; };
  // this warp's first neuron and its groups [gb, ge) of 8 blocks in a unit
  auto role = [&](int tile_, bool single, int hsel, int& nbase, int& gb, int& ge) {
    if (!single) {
      nbase = tile_ * kGrpNeurons + warp * kGrpNeuronsPerWarp;
      gb = 0;
      ge = nit;
    } else {
      nbase = tile_ * kGrpNeurons + hsel * (kGrpNeurons / 2) + (warp & 3) * kGrpNeuronsPerWarp;
      gb = warp < 4 ? 0 : half;
      ge = warp < 4 ? half : nit;
    }
  };

  auto load = [&](int e_, int nbase_, int it, GrpBuf<UNR>& U) {
    const size_t row = (size_t)e_ * I + nbase_ + g;
    const uint8_t* grow = gu_codes + row * 2 * H + q * 16;  // gate row, this lane's 16 B
    const uint8_t* urow = grow + H;
    const uint8_t* gsc = gu_scales + row * 2 * nblk;
    const uint8_t* usc = gsc + nblk;
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
  const uint8_t* xl = xs + g * RS;  // column g of tile 0
  const float zero[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  float* comb = reinterpret_cast<float*>(dsm + L.wc);  // free once the pairs are placed

  // the expert of item i: the last expert whose first item is at most i
  int e = 0;
  {
    const int i0 = item_of(u0);
    int lo = 0, hi = E - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_istart[mid] <= i0) lo = mid;
      else hi = mid - 1;
    }
    e = lo;
  }
  // the expert of item i, searched on from expert e
  auto expert_after = [&](int i, int e_) {
    while (e_ + 1 < E && s_istart[e_ + 1] <= i) ++e_;
    return e_;
  };
  GrpBuf<UNR> U0, U1;
  {  // the first codes, before any staging
    int nb, gb, ge;
    role((item_of(u0) - s_istart[e]) % tiles, is_single(u0), u0 & 1, nb, gb, ge);
    load(e, nb, gb, U0);
  }
  int staged_e = -1, staged_pass = -1;

  for (int u = u0; u < u1;) {
    const bool single = is_single(u);
    const int rem = item_of(u) - s_istart[e];
    const int pass = rem / tiles, tile = rem - pass * tiles;

    const int cols = min(kT, s_cnt[e] - pass * kT);
    if (e != staged_e || pass != staged_pass) {
      __syncthreads();  // every warp is done with the previous pass's columns
      // Stage the columns: warp c converts pair c's token row to f16 x 2^sigma.
      for (int c = warp; c < cols; c += kWarpsPerCta) {
        const int pr = s_list[s_start[e] + pass * kT + c];
        const int t = pr / top_k;
        const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H);
        float m = 0.0f;
        for (int k = lane; k < (H >> 3); k += 32) m = fmaxf(m, absmax8(ld_cached16(src + k)));
        const int sigma = pow2_shift_for(warp_max(m));
        const float up = exp2i(sigma);
        uint4* dst = reinterpret_cast<uint4*>(xs + (size_t)c * RS);
        for (int k = lane; k < (H >> 3); k += 32) dst[k] = to_f16x8(ld_cached16(src + k), up);
        if (lane == 0) {
          s_sig[c] = sigma;
          s_pair[c] = pr;
        }
      }
      __syncthreads();
      staged_e = e;
      staged_pass = pass;
    }
    int nbase, gb, ge;
    role(tile, single, u & 1, nbase, gb, ge);
    const int un = u + ((halves && !single) ? 2 : 1);  // the next unit

    // acc*: the running sum; lo*: the lower half of H's, once the upper half begins
    float accg[2], accu[2], lowg[2], lowu[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) accg[k] = accu[k] = lowg[k] = lowu[k] = 0.0f;
    auto stash = [&]() {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        lowg[k] = accg[k];
        lowu[k] = accu[k];
        accg[k] = accu[k] = 0.0f;
      }
    };

    auto compute = [&](int it, const GrpBuf<UNR>& U) {
#pragma unroll
      for (int i2 = 0; i2 < UNR / 2; ++i2) {
        // swap upper halves with lane q^2: each lane then holds 8 codes of both blocks
        const uint32_t rg2 = __shfl_xor_sync(kFull, U.g[i2].z, 2);
        const uint32_t rg3 = __shfl_xor_sync(kFull, U.g[i2].w, 2);
        const uint32_t ru2 = __shfl_xor_sync(kFull, U.u[i2].z, 2);
        const uint32_t ru3 = __shfl_xor_sync(kFull, U.u[i2].w, 2);
        const uint2 cgb[2] = {low ? make_uint2(U.g[i2].x, U.g[i2].y) : make_uint2(rg2, rg3),
                              low ? make_uint2(rg2, rg3) : make_uint2(U.g[i2].x, U.g[i2].y)};
        const uint2 cub[2] = {low ? make_uint2(U.u[i2].x, U.u[i2].y) : make_uint2(ru2, ru3),
                              low ? make_uint2(ru2, ru3) : make_uint2(U.u[i2].x, U.u[i2].y)};
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
          const int ib = 2 * i2 + hb;
          const int b = it * UNR + ib;
          uint32_t a0[4], a1[4];
          e4m3x4_to_f16x4(cgb[hb].x, a0[0], a0[2]);
          e4m3x4_to_f16x4(cub[hb].x, a0[1], a0[3]);
          e4m3x4_to_f16x4(cgb[hb].y, a1[0], a1[2]);
          e4m3x4_to_f16x4(cub[hb].y, a1[1], a1[3]);
          const uint32_t swd = (ib % 8) < 4 ? U.sg[ib / 8].x : U.sg[ib / 8].y;
          const uint32_t uwd = (ib % 8) < 4 ? U.su[ib / 8].x : U.su[ib / 8].y;
          float sg, su;
          e8m0x2_to_f32(swd >> (8 * (ib % 4)), uwd >> (8 * (ib % 4)), sg, su);
          const int off = hb ? off_odd : off_even;
          const uint4 xv = *reinterpret_cast<const uint4*>(xl + b * 64 + 2 * off);
          float d[4];
          mma_16816(d, a0, xv.x, xv.y, zero);
          mma_16816(d, a1, xv.z, xv.w, d);
          accg[0] = fmaf(d[0], sg, accg[0]);
          accg[1] = fmaf(d[1], sg, accg[1]);
          accu[0] = fmaf(d[2], su, accu[0]);
          accu[1] = fmaf(d[3], su, accu[1]);
        }
      }
    };

    // the next unit's first codes for this warp, into U0 once U0 is free
    auto load_next = [&]() {
      if (un < u1) {
        const int ni = item_of(un);
        const int en = expert_after(ni, e);
        int nb, b0, b1;
        role((ni - s_istart[en]) % tiles, is_single(un), un & 1, nb, b0, b1);
        load(en, nb, b0, U0);
      }
    };
    for (int it = gb; it < ge; it += 2) {
      if (it == half) stash();
      if (it + 1 < ge) {
        load(e, nbase, it + 1, U1);
        compute(it, U0);
        if (it + 2 < ge) load(e, nbase, it + 2, U0);
        else load_next();
        if (it + 1 == half) stash();
        compute(it + 1, U1);
      } else {  // an odd number of groups: the last one is in U0
        compute(it, U0);
        load_next();
      }
    }

    // The totals: lower partial + upper partial. A split half-item's upper
    // partials come from warps 4-7 through shared memory.
    bool writer = true;
    if (single) {
      float* cw = comb + ((warp & 3) * 32 + lane) * 4;
      if (warp >= 4) {
        cw[0] = accg[0];
        cw[1] = accg[1];
        cw[2] = accu[0];
        cw[3] = accu[1];
      }
      __syncthreads();
      writer = warp < 4;
      if (writer) {
        accg[0] += cw[0];
        accg[1] += cw[1];
        accu[0] += cw[2];
        accu[1] += cw[3];
      }
    } else {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        accg[k] = lowg[k] + accg[k];
        accu[k] = lowu[k] + accu[k];
      }
    }
    // Epilogue: lane (g, q) holds gate and up of neuron n for columns 2q, 2q+1.
    if (writer) {
      const int n = nbase + g;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int li = 2 * q + k;
        if (li < cols) {
          const float unscale = exp2i(-s_sig[li]);
          const float gv = accg[k] * unscale, uv = accu[k] * unscale;
          const float sl = gv / (1.0f + expf(-gv));
          const __nv_bfloat16 hv = __float2bfloat16_rn(sl * uv);
          h[(size_t)s_pair[li] * I + n] = *reinterpret_cast<const uint16_t*>(&hv);
        }
      }
    }
    if (single) __syncthreads();  // the combine buffer is free again
    if (un < u1) e = expert_after(item_of(un), e);
    u = un;
  }
}

template <int UNR>
moe_status launch_grouped(const moe_shape* s, const moe_weights* w, const uint16_t* x,
                          const int32_t* ids, int32_t B, uint16_t* h, int32_t* err,
                          cudaStream_t st, bool dependent) {
  const size_t smem = grp_layout(s->H, s->E, B * s->top_k).total;
  moe_status rc = allow_smem(moe_gate_up_grouped_kernel<UNR>, smem);
  if (rc != MOE_OK) return rc;
  const unsigned grid = (unsigned)(2 * sm_count());
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 1 : 0;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, moe_gate_up_grouped_kernel<UNR>, w->gu_codes,
                                           w->gu_scales, x, ids, h, err, s->H, s->I, s->E,
                                           s->top_k, B);
  if (e != cudaSuccess) {
    set_error("moe_gate_up_grouped launch", e);
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

constexpr int kGrpUnroll = 8;

}  // namespace

bool gate_up_grouped_supported(const moe_shape* s, const moe_weights* w, int32_t B) {
  return s->H % (32 * kGrpUnroll) == 0 && s->I % kGrpNeurons == 0 && s->E <= kThreads &&
         (w == nullptr || aligned(w->gu_scales, 8)) &&
         grp_layout(s->H, s->E, B * s->top_k).total <= kMaxDynSmem;
}

moe_status launch_gate_up_grouped(const moe_shape* s, const moe_weights* w, const uint16_t* x,
                                  const int32_t* ids, int32_t B, uint16_t* h, int32_t* err,
                                  cudaStream_t st, bool dependent) {
  // One column tile of 8 pairs per pass. Two tiles (16 staged rows, the codes
  // decoded once for both) were faster only from about 96 tokens of the
  // Qwen-3-30B-A3B shape while the kernel summed H in one chain; with the two
  // halves of H summed apart, their registers spilled and the one-tile form
  // with half-item shares is as fast or faster up to 128 tokens (96 tokens
  // 87.5 us against 101.3 for the two-tile form).
  return launch_grouped<kGrpUnroll>(s, w, x, ids, B, h, err, st, dependent);
}

}  // namespace wd
