// moe_down, expert-grouped form: one CTA per 16 output rows of y, for every
// token of the batch, streaming each routed expert's 16 down rows once.
//
// The per-token moe_down ("Better MoE model inference with warp decode",
// [§How the two kernels work]: each warp owns output dimensions of one token
// and streams the rows of all top-k experts into one FP32 accumulator with
// the routing weight folded in) decodes every down weight once per (token,
// slot) that uses it: at 32 tokens of the Qwen-3-30B-A3B shape, 403 M weight
// uses for 184 MB of unique weights. This form decodes each weight once per
// step and multiplies on the tensor cores, and still writes every y[t, o]
// once, from one CTA, with no atomics, no per-expert output buffer and no
// combine pass in global memory:
//
//   CTA c owns rows o0 = 16c .. o0+15 of y for all B tokens. The batch's
//   (token, slot) pairs are listed by expert, in pair order, and cut into
//   passes of up to 8 pairs of one expert; the CTA's 12 warps take the passes
//   in turn (pass j goes to warp j mod 12; with a few wide experts, each pass
//   is cut into chunks of its row and the warps take the chunks). For a pass
//   of expert e a warp
//   streams rows o0..o0+15 of e's down matrix (MMA rows 0..15) against the
//   intermediate rows of the pass's pairs (the MMA's 8 columns), one
//   mma.sync.m16n8k16 (f16 x f16 -> FP32) per 16 elements. Per 32-element
//   MXFP8 block the two MMAs' FP32 sums are multiplied by the row's E8M0
//   scale and added to an FP32 accumulator, as in the other kernels; after
//   the pass's last block, a lane's accumulator fragment (2 rows x 2 pairs)
//   is added, times each pair's routing weight, into the warp's own partial
//   sums of y for those rows and tokens, in shared memory. When every warp is
//   done, the CTA adds its 12 warps' partial sums in a fixed order and writes
//   each y[t, o] once. The sum over a token's experts is thereby split over
//   the CTA's warps (a reduction inside the CTA, in shared memory); the
//   per-token form keeps it inside one warp. Results are the same on every
//   call with the same inputs; a token's summation order depends on which
//   other tokens share the batch.
//
// Intermediate. The pairs' BF16 rows are copied into the warp's shared memory
// 256 elements at a time with cp.async and converted in place to
// f16 x 2^sigma, sigma chosen per (pair, 256 elements) from the largest
// magnitude so that it lies in [2^14, 2^15), the same rule as the per-token
// kernels; each step's sums are multiplied back by 2^-sigma per pair. The
// next step's codes (registers) and intermediate rows (the other shared
// buffer) are requested before this step computes.
//
// Measured on GB300 (one CTA per SM; 12 warps at 168 registers measured
// faster than 8 at 185 or 16 at 128): the kernel is bound by instruction
// issue and latency, not DRAM, so it pays only where experts are shared by
// several pairs (from about 3 pairs per expert); the layer uses it there.
//
// Loads. A quad of lanes reads 64 contiguous codes (two blocks) of one row;
// lanes q and q^2 swap their upper 8 codes, after which lane q holds 8 codes
// of each block at element offset 16(q&1) + 8(q>>1) (even block) or
// 16(q&1) + 8(1-(q>>1)) (odd block). The intermediate is read at the same
// offsets, so the k order inside a block is permuted identically for both
// operands and the sums are unchanged. A column's sums depend only on its own
// pair; which warp and column a pair lands in depends on the batch's routing.
//
// Duplicate ids (one token routed twice to an expert) fill two columns of the
// same token; their additions into the partial sums are made one lane group
// at a time. Pairs with an id outside [0, E) contribute nothing and set bit 0
// of the error flag.
#include "wd_device.cuh"
#include "wd_down_grouped.h"

namespace wd {
namespace {

constexpr int kDgRows = 16;                      // output rows per CTA (the MMA's M)
constexpr int kDgCols = 8;                       // pairs per pass (the MMA's N)
constexpr int kDgChunk = 256;                    // row elements per step (8 MXFP8 blocks)
constexpr int kDgColBytes = 2 * kDgChunk + 64;   // staged column stride: spreads banks
constexpr int kDgWarps = 12;                     // warps per CTA (one CTA per SM)
constexpr int kDgThreads = 32 * kDgWarps;
constexpr int kDgMaxE = 256;                     // the expert scan gives each thread one
constexpr int kDgMaxB = 128;

// Passes of up to 8 pairs: at most one partial pass per used expert.
__host__ __device__ inline int dg_max_passes(int E, int P) {
  return P / kDgCols + (E < P ? E : P);
}

// Byte offsets of the kernel's shared-memory arrays.
struct DgLayout {
  size_t h, sig, y, list, tok, wt, cnt, start, pstart, run, wc, pass, nused, total;
};

__host__ __device__ inline DgLayout dg_layout(int E, int P, int B) {
  DgLayout L;
  size_t o = 0;
  L.h = o;       // [warp][2 buffers][8 columns] x kDgColBytes: staged intermediate
  o += (size_t)kDgWarps * 2 * kDgCols * kDgColBytes;
  L.sig = o;     // [warp][2][8] int: its scale exponents
  o += (size_t)kDgWarps * 2 * kDgCols * 4;
  L.y = o;       // [warp][B][16] float: each warp's partial sums of y
  o += (size_t)kDgWarps * B * kDgRows * 4;
  L.list = o;    // [P] int: pair indices grouped by expert, in pair order
  o += (size_t)P * 4;
  L.tok = o;     // [P] int: their tokens
  o += (size_t)P * 4;
  L.wt = o;      // [P] float: their routing weights
  o += (size_t)P * 4;
  L.cnt = o;     // [E] int: pairs routed to each expert
  o += (size_t)E * 4;
  L.start = o;   // [E] int: first list entry of each expert
  o += (size_t)E * 4;
  L.pstart = o;  // [E] int: first pass (8 pairs each) of each expert
  o += (size_t)E * 4;
  L.run = o;     // [E] int: entries placed so far
  o += (size_t)E * 4;
  L.wc = o;      // [warp][E] int: per-warp counts while placing
  o += (size_t)kDgWarps * E * 4;
  o = (o + 15) & ~(size_t)15;
  L.pass = o;    // [passes] int4 (16-byte aligned): expert, first list entry, pairs,
                 // duplicate token
  o += (size_t)dg_max_passes(E, P) * 16;
  L.nused = o;   // int: number of passes
  o += 16;
  L.total = o;
  return L;
}

struct DgBuf {
  uint4 r0[4], r1[4];  // this lane's 16 codes of the step's 4 block pairs: row g, row g+8
  uint2 s0, s1;        // the E8M0 scales of the step's 8 blocks: row g, row g+8
};


__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
// Waits for this thread's own earlier copies (all but the N most recent groups).
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// The largest exponent field among 8 BF16 values.
__device__ __forceinline__ uint32_t bf16x8_max_exp(const uint4& v) {
  const uint32_t m = __vmaxu2(__vmaxu2(v.x & 0x7F807F80u, v.y & 0x7F807F80u),
                              __vmaxu2(v.z & 0x7F807F80u, v.w & 0x7F807F80u));
  return max(m & 0xFFFFu, m >> 16) >> 7;
}

// sigma for values whose largest BF16 exponent field is ex: the largest
// magnitude m has 2^(ex-127) <= m < 2^(ex-126), so m * 2^(141-ex) lies in
// [2^14, 2^15) (the rule of the per-token kernels). 126 for zero or subnormal
// values, 0 when an Inf or NaN is among them.
__device__ __forceinline__ int sigma_from_exp(uint32_t ex) {
  if (ex == 255u) return 0;
  if (ex == 0u) return 126;
  return min(126, max(-126, 141 - (int)ex));
}

__global__ void __launch_bounds__(kDgThreads, 1)
    moe_down_grouped_kernel(const uint8_t* __restrict__ d_codes,
                            const uint8_t* __restrict__ d_scales,
                            const uint16_t* __restrict__ h, const int32_t* __restrict__ ids,
                            const float* __restrict__ wts, float* __restrict__ y,
                            int32_t* __restrict__ err, int H, int I, int E, int top_k, int B) {
  extern __shared__ __align__(16) uint8_t dsm[];
  __shared__ int s_wtot[2][kDgWarps];
  const int P = B * top_k;
  const DgLayout L = dg_layout(E, P, B);
  uint8_t* s_h = dsm + L.h;
  int* s_sig = reinterpret_cast<int*>(dsm + L.sig);
  float* s_y = reinterpret_cast<float*>(dsm + L.y);
  int* s_list = reinterpret_cast<int*>(dsm + L.list);
  int* s_tok = reinterpret_cast<int*>(dsm + L.tok);
  float* s_wt = reinterpret_cast<float*>(dsm + L.wt);
  int* s_cnt = reinterpret_cast<int*>(dsm + L.cnt);
  int* s_start = reinterpret_cast<int*>(dsm + L.start);
  int* s_pstart = reinterpret_cast<int*>(dsm + L.pstart);
  int* s_run = reinterpret_cast<int*>(dsm + L.run);
  int* s_wc = reinterpret_cast<int*>(dsm + L.wc);
  int* s_nused = reinterpret_cast<int*>(dsm + L.nused);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, q = lane & 3;  // MMA group (row g and g+8) and lane in the quad
  const int o0 = blockIdx.x * kDgRows;
  const int nblk = I >> 5;
  constexpr unsigned kFull = 0xFFFFFFFFu;

  // ---- pair lists by expert (ids and routing weights are layer inputs: all of
  // this runs before the wait for the intermediate) ----
  for (int i = tid; i < E; i += kDgThreads) {
    s_cnt[i] = 0;
    s_run[i] = 0;
  }
  for (int i = tid; i < kDgWarps * E; i += kDgThreads) s_wc[i] = 0;
  for (int i = tid; i < kDgWarps * B * kDgRows; i += kDgThreads) s_y[i] = 0.0f;
  __syncthreads();
  bool bad = false;
  for (int p = tid; p < P; p += kDgThreads) {
    const int e = __ldg(ids + p);
    if (e >= 0 && e < E) atomicAdd(s_cnt + e, 1);
    else bad = true;
  }
  __syncthreads();
  {  // exclusive scans over the experts (one per thread): list offsets and
     // pass offsets
    const int c = tid < E ? s_cnt[tid] : 0;
    const int np = (c + kDgCols - 1) / kDgCols;
    int ic = c, ip = np;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int a = __shfl_up_sync(kFull, ic, d), b = __shfl_up_sync(kFull, ip, d);
      if (lane >= d) {
        ic += a;
        ip += b;
      }
    }
    if (lane == 31) {
      s_wtot[0][warp] = ic;
      s_wtot[1][warp] = ip;
    }
    __syncthreads();
    int bc = 0, bp = 0;
    for (int w = 0; w < warp; ++w) {
      bc += s_wtot[0][w];
      bp += s_wtot[1][w];
    }
    if (tid < E) {
      s_start[tid] = bc + ic - c;
      s_pstart[tid] = bp + ip - np;
    }
    if (tid == kDgThreads - 1) *s_nused = bp + ip;
  }
  __syncthreads();
  // Place the pairs in pair order: within a warp by match, across warps by the
  // warps' counts of the same expert, across rounds by the running count.
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int c0 = 0; c0 < P; c0 += kDgThreads) {
    const int p = c0 + tid;
    const int e = p < P ? __ldg(ids + p) : -1;
    const bool valid = e >= 0 && e < E;
    const unsigned m = __match_any_sync(kFull, valid ? e : -1);
    const int lt = __popc(m & lt_mask);
    if (valid && lt == 0) s_wc[warp * E + e] = __popc(m);
    __syncthreads();
    if (valid) {
      int r = s_run[e] + lt;
      for (int w = 0; w < warp; ++w) r += s_wc[w * E + e];
      const int idx = s_start[e] + r;
      s_list[idx] = p;
      s_tok[idx] = p / top_k;
      s_wt[idx] = __ldg(wts + p);
    }
    __syncthreads();
    if (valid && lt == 0) {
      atomicAdd(s_run + e, __popc(m));
      s_wc[warp * E + e] = 0;
    }
    __syncthreads();
  }
  // Pass table: pass j of expert e covers list entries start + 8j .. (at most
  // 8); .w is 1 if two of its pairs share a token (a duplicate id).
  int4* s_pass = reinterpret_cast<int4*>(dsm + L.pass);
  for (int e = tid; e < E; e += kDgThreads) {
    const int c = s_cnt[e];
    for (int j = 0; j * kDgCols < c; ++j) {
      const int base = s_start[e] + j * kDgCols, n = min(kDgCols, c - j * kDgCols);
      int dup = 0;
      for (int k = 1; k < n; ++k) dup |= s_tok[base + k] == s_tok[base + k - 1];
      s_pass[s_pstart[e] + j] = make_int4(e, base, n, dup);
    }
  }
  __syncthreads();
  const int npass = *s_nused;
  const int nck = I / kDgChunk;
  // Work items: a pass, or, when the CTA has fewer than 6 passes per warp
  // (few wide experts, e.g. Mixtral-shaped I = 14336 with 16 passes per CTA),
  // chunks of at least 4 of its steps, up to about 12 items per warp; each
  // item's sums are added into the partial y of the warp that ran it.
  // Measured on GB300: shorter or uneven chunks, or chunks where passes are
  // many, cost more in per-item work than they gain in balance.
  const int want = (12 * kDgWarps + npass - 1) / max(npass, 1);
  const int parts = npass < 6 * kDgWarps ? max(1, min(want, nck / 4)) : 1;
  const int spc = (nck + parts - 1) / parts;        // steps per item
  const int nch = (nck + spc - 1) / spc;            // items per pass
  const int nitem = npass * nch;

  // ---- the warp's items (a pass of up to 8 pairs of one expert, or a chunk
  // of it): warp, warp + kDgWarps, ...; each in steps of 256 row elements ----
  uint8_t* my_h = s_h + (size_t)warp * 2 * kDgCols * kDgColBytes;
  int* my_sig = s_sig + warp * 2 * kDgCols;
  float* my_y = s_y + (size_t)warp * B * kDgRows;

  auto wload = [&](int e, int kc, DgBuf& W) {
    const size_t row = (size_t)e * H + o0 + g;
    const uint8_t* c0p = d_codes + row * I + (size_t)kc * kDgChunk + q * 16;
    const uint8_t* c1p = c0p + (size_t)8 * I;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      W.r0[i] = ld_codes16(c0p + 64 * i);
      W.r1[i] = ld_codes16(c1p + 64 * i);
    }
    const uint8_t* sp = d_scales + row * nblk + kc * 8;
    W.s0 = ld_scales8(sp);
    W.s1 = ld_scales8(sp + (size_t)8 * nblk);
  };
  // the pass's intermediate rows for one step, copied into buffer b
  auto hload = [&](const int4& ps, int kc, int b) {
    uint8_t* dst = my_h + (size_t)b * kDgCols * kDgColBytes + 16 * lane;
    const uint16_t* src = h + (size_t)kc * kDgChunk + 8 * lane;
    for (int k = 0; k < ps.z; ++k)
      cp_async16(dst + k * kDgColBytes, src + (size_t)s_list[ps.y + k] * I);
    cp_async_commit();
  };
  auto hconvert = [&](int n, int b) {
    uint8_t* base = my_h + (size_t)b * kDgCols * kDgColBytes + 16 * lane;
    for (int c = 0; c < n; ++c) {
      uint4* ptr = reinterpret_cast<uint4*>(base + c * kDgColBytes);
      const uint4 v = *ptr;
      const int sigma = sigma_from_exp(__reduce_max_sync(kFull, bf16x8_max_exp(v)));
      *ptr = to_f16x8(v, exp2i(sigma));
      if (lane == 0) my_sig[b * kDgCols + c] = sigma;
    }
  };

  float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  const int off_even = 16 * (q & 1) + 8 * (q >> 1);
  const int off_odd = 16 * (q & 1) + 8 * (1 - (q >> 1));
  const bool low = q < 2;
  auto compute = [&](const DgBuf& W, int b) {
    const uint8_t* hc = my_h + ((size_t)b * kDgCols + g) * kDgColBytes;
    float sc0[8], sc1[8];  // the step's block scales of rows g and g+8
    {
      float t[4];
      e8m0x4_to_f32(W.s0.x, t);
#pragma unroll
      for (int i = 0; i < 4; ++i) sc0[i] = t[i];
      e8m0x4_to_f32(W.s0.y, t);
#pragma unroll
      for (int i = 0; i < 4; ++i) sc0[4 + i] = t[i];
      e8m0x4_to_f32(W.s1.x, t);
#pragma unroll
      for (int i = 0; i < 4; ++i) sc1[i] = t[i];
      e8m0x4_to_f32(W.s1.y, t);
#pragma unroll
      for (int i = 0; i < 4; ++i) sc1[4 + i] = t[i];
    }
    float cacc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    const float zero[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int i2 = 0; i2 < 4; ++i2) {
      // swap upper halves with lane q^2: each lane then holds 8 codes of both blocks
      const uint32_t x2 = __shfl_xor_sync(kFull, W.r0[i2].z, 2);
      const uint32_t x3 = __shfl_xor_sync(kFull, W.r0[i2].w, 2);
      const uint32_t z2 = __shfl_xor_sync(kFull, W.r1[i2].z, 2);
      const uint32_t z3 = __shfl_xor_sync(kFull, W.r1[i2].w, 2);
      const uint2 ra[2] = {low ? make_uint2(W.r0[i2].x, W.r0[i2].y) : make_uint2(x2, x3),
                           low ? make_uint2(x2, x3) : make_uint2(W.r0[i2].x, W.r0[i2].y)};
      const uint2 rb[2] = {low ? make_uint2(W.r1[i2].x, W.r1[i2].y) : make_uint2(z2, z3),
                           low ? make_uint2(z2, z3) : make_uint2(W.r1[i2].x, W.r1[i2].y)};
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) {
        const int bi = 2 * i2 + hb;  // block of the step
        uint32_t a0[4], a1[4];
        e4m3x4_to_f16x4(ra[hb].x, a0[0], a0[2]);
        e4m3x4_to_f16x4(rb[hb].x, a0[1], a0[3]);
        e4m3x4_to_f16x4(ra[hb].y, a1[0], a1[2]);
        e4m3x4_to_f16x4(rb[hb].y, a1[1], a1[3]);
        const int off = hb ? off_odd : off_even;
        const uint4 xv = *reinterpret_cast<const uint4*>(hc + (bi * 32 + off) * 2);
        float d[4];
        mma_16816(d, a0, xv.x, xv.y, zero);
        mma_16816(d, a1, xv.z, xv.w, d);
        cacc[0] = fmaf(d[0], sc0[bi], cacc[0]);
        cacc[1] = fmaf(d[1], sc0[bi], cacc[1]);
        cacc[2] = fmaf(d[2], sc1[bi], cacc[2]);
        cacc[3] = fmaf(d[3], sc1[bi], cacc[3]);
      }
    }
    // columns 2q, 2q+1 back from their staging scales (columns beyond the
    // pass's pairs hold stale values that are never used)
    const float u0 = exp2i(-my_sig[b * kDgCols + 2 * q]);
    const float u1 = exp2i(-my_sig[b * kDgCols + 2 * q + 1]);
    acc[0] = fmaf(cacc[0], u0, acc[0]);
    acc[1] = fmaf(cacc[1], u1, acc[1]);
    acc[2] = fmaf(cacc[2], u0, acc[2]);
    acc[3] = fmaf(cacc[3], u1, acc[3]);
  };
  // End of a pass: add routing weight x sums into the warp's partial y. Two
  // columns of one token (a duplicate id) can sit in different lanes; then
  // the lanes add one quad position at a time.
  auto flush = [&](const int4& ps) {
    const int n = ps.z, base = ps.y;
    auto add = [&]() {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int cc = 2 * q + k;
        if (cc < n) {
          const float wv = s_wt[base + cc];
          float* yt = my_y + (size_t)s_tok[base + cc] * kDgRows;
          yt[g] = fmaf(wv, acc[k], yt[g]);
          yt[g + 8] = fmaf(wv, acc[2 + k], yt[g + 8]);
        }
      }
    };
    if (!ps.w) {
      add();
    } else {
#pragma unroll
      for (int ph = 0; ph < 4; ++ph) {
        if (q == ph) add();
        __syncwarp();
      }
    }
    __syncwarp();
    acc[0] = acc[1] = acc[2] = acc[3] = 0.0f;
  };

  // Pipeline: step k computes from register buffer k % 2 and shared buffer
  // k % 2; the codes and intermediate rows of step k + 1 are requested at its
  // start into the other buffers.
  auto item_k0 = [&](int i) { return (i - (i / nch) * nch) * spc; };
  int it = warp, kc = 0;  // the warp's current item and step
  DgBuf W0, W1;
  if (it < nitem) {  // the first codes, before the wait
    kc = item_k0(it);
    wload(s_pass[it / nch].x, kc, W0);
  }
  wait_prerequisite();  // the intermediate h is complete from here on
  if (it < nitem) {
    int4 ps = s_pass[it / nch];
    int kend = min(nck, kc + spc);
    hload(ps, kc, 0);
    int buf = 0;
    auto step = [&](DgBuf& Wc, DgBuf& Wn) -> bool {
      int in = it, kn = kc + 1, kendn = kend;
      const bool last = kn == kend;  // this step ends the item
      if (last) in = it + kDgWarps;
      const bool more = in < nitem;
      int4 nps = ps;
      if (last && more) {
        nps = s_pass[in / nch];
        kn = item_k0(in);
        kendn = min(nck, kn + spc);
      }
      __syncwarp();  // every lane has finished reading the buffers being refilled
      if (more) {
        wload(nps.x, kn, Wn);
        hload(nps, kn, buf ^ 1);
        cp_async_wait<1>();
      } else {
        cp_async_wait<0>();
      }
      __syncwarp();
      hconvert(ps.z, buf);
      __syncwarp();
      compute(Wc, buf);
      if (last) flush(ps);
      it = in;
      kc = kn;
      kend = kendn;
      ps = nps;
      buf ^= 1;
      return more;
    };
    while (step(W0, W1) && step(W1, W0)) {
    }
  }
  if (bad) flag_invalid(err);

  // ---- every y[t, o0..o0+15]: the warps' partial sums in warp order ----
  __syncthreads();
  for (int i = tid; i < B * kDgRows; i += kDgThreads) {
    const int t = i / kDgRows, r = i - t * kDgRows;
    float v = 0.0f;
#pragma unroll
    for (int w = 0; w < kDgWarps; ++w) v += s_y[((size_t)w * B + t) * kDgRows + r];
    y[(size_t)t * H + o0 + r] = v;
  }
}

}  // namespace

bool down_grouped_supported(const moe_shape* s, const moe_weights* w, int32_t B) {
  if (s->I % kDgChunk || s->H % kDgRows || s->E > kDgMaxE || B < 1 || B > kDgMaxB) return false;
  if (w && !aligned(w->d_scales, 8)) return false;
  return dg_layout(s->E, B * s->top_k, B).total <= kMaxDynSmem;
}

moe_status launch_down_grouped(const moe_shape* s, const moe_weights* w, const uint16_t* h,
                               const int32_t* ids, const float* wts, int32_t B, float* y,
                               int32_t* err, cudaStream_t st, bool dependent) {
  const size_t smem = dg_layout(s->E, B * s->top_k, B).total;
  moe_status rc = allow_smem(moe_down_grouped_kernel, smem);
  if (rc != MOE_OK) return rc;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(s->H / kDgRows));
  cfg.blockDim = dim3(kDgThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 1 : 0;
  const cudaError_t e =
      cudaLaunchKernelEx(&cfg, moe_down_grouped_kernel, w->d_codes, w->d_scales, h, ids, wts, y,
                         err, s->H, s->I, s->E, s->top_k, B);
  if (e != cudaSuccess) {
    set_error("moe_down_grouped launch", e);
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

}  // namespace wd
