/*
 * CPU ORACLE for the output-centric ("warp decode") MoE decode layer.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this code; the product path never does. It shares
 * no code with the CUDA path: everything below is written out from the
 * definitions, in double precision, single-threaded, with no blocking, fusion
 * or reordering beyond what the definitions state.
 *
 * What the layer computes ("Better MoE model inference with warp decode",
 * Key claims [§Reorganized parallelism], [§How the two kernels work] and the
 * Method section; sd114.wiki "Warp Decode" page, section
 * 技术原理：两个 Kernel 搞定一切):
 *
 *   for each token t and each routed slot j (expert e = ids[t,j]):
 *     g[n] = sum_h x[t,h] * Wg[e,n,h]         (gate projection)
 *     u[n] = sum_h x[t,h] * Wu[e,n,h]         (up projection, same read of x)
 *     h[n] = bf16( silu(g[n]) * u[n] )        (SwiGLU, intermediate written out
 *                                              in BF16: activations stay BF16)
 *   y[t,o] = sum_j w[t,j] * sum_i h_j[i] * Wd[e_j,o,i]
 *                                             (down projection with the routing
 *                                              weight folded into one sum)
 *
 * The warp-decode method reaches exactly this result (it re-associates the
 * top-k combination, which is linear), so the oracle is the definition itself.
 *
 * Weights are MXFP8 (OCP Microscaling Formats v1.0): E4M3 element codes with
 * one E8M0 scale per 32 consecutive elements along the reduction axis
 * (H for gate/up, I for down). Canonical layouts used here:
 *   gate/up codes [E][I][H], scales [E][I][H/32]
 *   down    codes [E][H][I], scales [E][H][I/32]
 *
 * Readings where the pages are silent (each listed in the design notes):
 *  - SiLU(g) = g / (1 + exp(-g)); SwiGLU = SiLU(gate) * up, no biases.
 *  - The intermediate is rounded once to BF16, round-to-nearest-even, from the
 *    exact (here: double) value of SiLU(g)*u.
 *  - The routing weight multiplies the down projection of the BF16
 *    intermediate; the output y is FP32-or-wider (double here).
 *  - A slot whose expert id is outside [0, E) contributes nothing and its
 *    intermediate is 0; the count of such slots is returned.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------- MXFP8 element and scale decoding (OCP MX v1.0) ---------------- */

/* E4M3 ("E4M3FN"): 1 sign, 4 exponent (bias 7), 3 mantissa bits.
 * exponent 0: subnormal, value = (m/8) * 2^-6. Otherwise (1 + m/8) * 2^(e-7).
 * No infinities; S.1111.111 is NaN. Largest finite magnitude 448. */
double oracle_e4m3_value(uint8_t code) {
  int sign = (code >> 7) & 1;
  int e = (code >> 3) & 0xF;
  int m = code & 0x7;
  double mag;
  if (e == 0xF && m == 0x7) return NAN;
  if (e == 0)
    mag = ldexp((double)m / 8.0, -6);
  else
    mag = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -mag : mag;
}

/* E8M0 scale: 2^(s - 127); 0xFF is NaN. */
double oracle_e8m0_value(uint8_t s) {
  if (s == 0xFF) return NAN;
  return ldexp(1.0, (int)s - 127);
}

/* Value tables filled once from the two functions above, so that the layer
 * loops do not recompute ldexp for every element. */
static double e4m3_table[256], e8m0_table[256];
static int tables_ready = 0;

static void fill_tables(void) {
  if (tables_ready) return;
  for (int c = 0; c < 256; ++c) {
    e4m3_table[c] = oracle_e4m3_value((uint8_t)c);
    e8m0_table[c] = oracle_e8m0_value((uint8_t)c);
  }
  tables_ready = 1;
}

/* One MXFP8 element: code value times its block's scale. */
static double mx_element(uint8_t code, uint8_t scale) {
  return e4m3_table[code] * e8m0_table[scale];
}

/* ---------- BF16 ------------------------------------------------------------ */

double oracle_bf16_value(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Nearest BF16 to v, ties to the even significand. Written from the
 * definition: v lies between two adjacent BF16 values a <= v <= b; return the
 * closer one (the one with an even last bit on a tie). NaN -> 0x7FC0. */
uint16_t oracle_bf16_rne(double v) {
  if (isnan(v)) return 0x7FC0;
  uint16_t sign = signbit(v) ? 0x8000 : 0;
  double a = fabs(v);
  /* Largest BF16 finite value: (2 - 2^-7) * 2^127. Values at or beyond the
   * midpoint between it and 2^128 round to infinity. */
  double maxf = ldexp(2.0 - ldexp(1.0, -7), 127);
  double overflow_mid = ldexp(2.0 - ldexp(1.0, -8), 127);
  if (a >= overflow_mid) return (uint16_t)(sign | 0x7F80);
  if (a >= maxf) return (uint16_t)(sign | 0x7F7F);
  /* Magnitude codes 0x0000..0x7F7F are increasing in value: binary search
   * for the largest code whose value is <= a. */
  int lo = 0, hi = 0x7F7F;
  while (lo < hi) {
    int mid = (lo + hi + 1) / 2;
    if (oracle_bf16_value((uint16_t)mid) <= a)
      lo = mid;
    else
      hi = mid - 1;
  }
  double below = oracle_bf16_value((uint16_t)lo);
  if (below == a) return (uint16_t)(sign | lo);
  double above = oracle_bf16_value((uint16_t)(lo + 1));
  double d_lo = a - below, d_hi = above - a;
  int pick;
  if (d_lo < d_hi)
    pick = lo;
  else if (d_hi < d_lo)
    pick = lo + 1;
  else
    pick = (lo & 1) ? lo + 1 : lo;
  return (uint16_t)(sign | pick);
}

/* ---------- SwiGLU ---------------------------------------------------------- */

double oracle_silu(double g) { return g / (1.0 + exp(-g)); }

/* ---------- MXFP8 quantiser (OCP MX v1.0, section "Conversion") ------------
 * For each block of 32 consecutive FP32 values V along a row:
 *   shared_exp = floor(log2(max|V|)) - 8     (8 = exponent of E4M3's largest
 *                                             normal, 448 = 1.75 * 2^8)
 *   X = 2^shared_exp, stored as the E8M0 code shared_exp + 127, clamped to
 *   [0, 254]; a block of zeros stores code 0.
 *   P_i = V_i / X rounded to the nearest E4M3 value, ties to even code,
 *   magnitudes above 448 clamped to 448.
 * rows x K values in, rows x K codes and rows x (K/32) scales out. K % 32 == 0.
 */
static uint8_t e4m3_nearest(double v) {
  if (isnan(v)) return 0x7F;
  uint8_t sign = signbit(v) ? 0x80 : 0;
  double a = fabs(v);
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);
  /* codes 0x00..0x7E have increasing magnitude */
  int lo = 0, hi = 0x7E;
  while (lo < hi) {
    int mid = (lo + hi + 1) / 2;
    if (e4m3_table[mid] <= a)
      lo = mid;
    else
      hi = mid - 1;
  }
  double below = e4m3_table[lo];
  if (below == a) return (uint8_t)(sign | lo);
  double above = e4m3_table[lo + 1];
  double d_lo = a - below, d_hi = above - a;
  int pick;
  if (d_lo < d_hi)
    pick = lo;
  else if (d_hi < d_lo)
    pick = lo + 1;
  else
    pick = (lo & 1) ? lo + 1 : lo;
  return (uint8_t)(sign | pick);
}

int oracle_quantize_mxfp8(const float* w, int64_t rows, int64_t K, uint8_t* codes,
                          uint8_t* scales) {
  if (K % 32 != 0 || rows < 0) return -1;
  fill_tables();
  int64_t nb = K / 32;
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t b = 0; b < nb; ++b) {
      const float* v = w + r * K + b * 32;
      double amax = 0.0;
      for (int i = 0; i < 32; ++i) {
        double a = fabs((double)v[i]);
        if (a > amax) amax = a;
      }
      int s;
      if (amax == 0.0) {
        s = 0;
      } else if (isinf(amax)) {
        s = 254;
      } else {
        int ex;
        frexp(amax, &ex); /* amax = f * 2^ex, f in [0.5, 1): floor(log2) = ex-1 */
        int shared_exp = (ex - 1) - 8;
        s = shared_exp + 127;
        if (s < 0) s = 0;
        if (s > 254) s = 254;
      }
      scales[r * nb + b] = (uint8_t)s;
      double X = ldexp(1.0, s - 127);
      for (int i = 0; i < 32; ++i)
        codes[r * K + b * 32 + i] = e4m3_nearest((double)v[i] / X);
    }
  }
  return 0;
}

/* Decode a whole MXFP8 matrix (rows x K) into doubles (for the tests). */
int oracle_dequantize_mxfp8(const uint8_t* codes, const uint8_t* scales, int64_t rows,
                            int64_t K, double* out) {
  if (K % 32 != 0 || rows < 0) return -1;
  fill_tables();
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t k = 0; k < K; ++k)
      out[r * K + k] = mx_element(codes[r * K + k], scales[r * (K / 32) + k / 32]);
  return 0;
}

/* ---------- The MoE decode layer -------------------------------------------
 * x       [B][H]   BF16 bits
 * ids     [B][k]   expert ids
 * wts     [B][k]   routing weights (FP32)
 * gate/up codes [E][I][H], scales [E][I][H/32]; down codes [E][H][I], scales
 * [E][H][I/32]
 * y       [B][H]   output (double), overwritten
 * h_out   [B][k][I] BF16 bits of the intermediate, or NULL
 * Returns the number of slots whose id was outside [0, E), or -1 on bad shape.
 */
int64_t oracle_moe_layer(int32_t H, int32_t I, int32_t E, int32_t k, int32_t B,
                         const uint16_t* x, const int32_t* ids, const float* wts,
                         const uint8_t* gate_codes, const uint8_t* gate_scales,
                         const uint8_t* up_codes, const uint8_t* up_scales,
                         const uint8_t* down_codes, const uint8_t* down_scales,
                         double* y, uint16_t* h_out) {
  if (H <= 0 || I <= 0 || E <= 0 || k <= 0 || B < 0 || H % 32 || I % 32) return -1;
  fill_tables();
  int64_t invalid = 0;
  const int64_t hb = H / 32, ib = I / 32;
  double* xval = (double*)malloc(sizeof(double) * (size_t)H);  /* x[t,:] as values */
  double* hval = (double*)malloc(sizeof(double) * (size_t)I);  /* BF16 intermediate */
  uint16_t* hbits = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)I);
  if (!xval || !hval || !hbits) {
    free(xval);
    free(hval);
    free(hbits);
    return -1;
  }
  for (int32_t t = 0; t < B; ++t) {
    const uint16_t* xt = x + (int64_t)t * H;
    for (int32_t hh = 0; hh < H; ++hh) xval[hh] = oracle_bf16_value(xt[hh]);
    double* yt = y + (int64_t)t * H;
    for (int32_t o = 0; o < H; ++o) yt[o] = 0.0;
    for (int32_t j = 0; j < k; ++j) {
      int32_t e = ids[(int64_t)t * k + j];
      uint16_t* hdst = h_out ? h_out + ((int64_t)t * k + j) * I : NULL;
      if (e < 0 || e >= E) {
        ++invalid;
        if (hdst) memset(hdst, 0, sizeof(uint16_t) * (size_t)I);
        continue;
      }
      /* gate / up projections and SwiGLU, one intermediate neuron at a time */
      for (int32_t n = 0; n < I; ++n) {
        int64_t row = (int64_t)e * I + n;
        double g = 0.0, u = 0.0;
        for (int32_t hh = 0; hh < H; ++hh) {
          double xv = xval[hh];
          g += xv * mx_element(gate_codes[row * H + hh], gate_scales[row * hb + hh / 32]);
          u += xv * mx_element(up_codes[row * H + hh], up_scales[row * hb + hh / 32]);
        }
        hbits[n] = oracle_bf16_rne(oracle_silu(g) * u);
        hval[n] = oracle_bf16_value(hbits[n]);
      }
      if (hdst) memcpy(hdst, hbits, sizeof(uint16_t) * (size_t)I);
      /* down projection of this slot, weighted, added into y */
      double wj = (double)wts[(int64_t)t * k + j];
      for (int32_t o = 0; o < H; ++o) {
        int64_t row = (int64_t)e * H + o;
        double acc = 0.0;
        for (int32_t i = 0; i < I; ++i)
          acc += hval[i] * mx_element(down_codes[row * I + i], down_scales[row * ib + i / 32]);
        yt[o] += wj * acc;
      }
    }
  }
  free(xval);
  free(hval);
  free(hbits);
  return invalid;
}

/* ---------- Variants for the accuracy study --------------------------------
 * "Better MoE model inference with warp decode", Key claims [§Improved
 * accuracy] (and the sd114.wiki page, 性能与精度双重提升, item 2): the
 * conventional path quantises each BF16 activation to MXFP8 before a
 * projection and back (a BF16 -> MXFP8 -> BF16 round trip); warp decode keeps
 * activations in BF16 with FP32 accumulators, and its output is reported
 * closer to a full-precision reference.
 *
 * The same layer as oracle_moe_layer, with two switches:
 *   round_h : 1 = the intermediate is rounded to BF16 (the layer's own rule),
 *             0 = it is kept exact (a full-precision reference);
 *   mx_acts : 1 = the activation entering each projection (x for gate/up, the
 *             intermediate for down) is first replaced by its MXFP8 round
 *             trip (OCP MX v1.0 conversion, as in oracle_quantize_mxfp8);
 *             0 = it is used as is.
 * oracle_moe_layer equals round_h = 1, mx_acts = 0. y [B][H] is written;
 * returns the number of out-of-range slots, or -1 on a bad shape.
 */
static void mx_roundtrip(double* v, int64_t K) {
  for (int64_t b = 0; b < K / 32; ++b) {
    double* blk = v + b * 32;
    double amax = 0.0;
    for (int i = 0; i < 32; ++i)
      if (fabs(blk[i]) > amax) amax = fabs(blk[i]);
    int s;
    if (amax == 0.0) {
      s = 0;
    } else if (isinf(amax)) {
      s = 254;
    } else {
      int ex;
      frexp(amax, &ex);
      s = (ex - 1) - 8 + 127;
      if (s < 0) s = 0;
      if (s > 254) s = 254;
    }
    double X = ldexp(1.0, s - 127);
    for (int i = 0; i < 32; ++i) blk[i] = e4m3_table[e4m3_nearest(blk[i] / X)] * X;
  }
}

int64_t oracle_moe_layer_variant(int32_t H, int32_t I, int32_t E, int32_t k, int32_t B,
                                 const uint16_t* x, const int32_t* ids, const float* wts,
                                 const uint8_t* gate_codes, const uint8_t* gate_scales,
                                 const uint8_t* up_codes, const uint8_t* up_scales,
                                 const uint8_t* down_codes, const uint8_t* down_scales,
                                 int32_t round_h, int32_t mx_acts, double* y) {
  if (H <= 0 || I <= 0 || E <= 0 || k <= 0 || B < 0 || H % 32 || I % 32) return -1;
  fill_tables();
  int64_t invalid = 0;
  const int64_t hb = H / 32, ib = I / 32;
  double* xval = (double*)malloc(sizeof(double) * (size_t)H);
  double* hval = (double*)malloc(sizeof(double) * (size_t)I);
  if (!xval || !hval) {
    free(xval);
    free(hval);
    return -1;
  }
  for (int32_t t = 0; t < B; ++t) {
    for (int32_t hh = 0; hh < H; ++hh) xval[hh] = oracle_bf16_value(x[(int64_t)t * H + hh]);
    if (mx_acts) mx_roundtrip(xval, H);
    double* yt = y + (int64_t)t * H;
    for (int32_t o = 0; o < H; ++o) yt[o] = 0.0;
    for (int32_t j = 0; j < k; ++j) {
      int32_t e = ids[(int64_t)t * k + j];
      if (e < 0 || e >= E) {
        ++invalid;
        continue;
      }
      for (int32_t n = 0; n < I; ++n) {
        int64_t row = (int64_t)e * I + n;
        double g = 0.0, u = 0.0;
        for (int32_t hh = 0; hh < H; ++hh) {
          g += xval[hh] * mx_element(gate_codes[row * H + hh], gate_scales[row * hb + hh / 32]);
          u += xval[hh] * mx_element(up_codes[row * H + hh], up_scales[row * hb + hh / 32]);
        }
        double hv = oracle_silu(g) * u;
        hval[n] = round_h ? oracle_bf16_value(oracle_bf16_rne(hv)) : hv;
      }
      if (mx_acts) mx_roundtrip(hval, I);
      double wj = (double)wts[(int64_t)t * k + j];
      for (int32_t o = 0; o < H; ++o) {
        int64_t row = (int64_t)e * H + o;
        double acc = 0.0;
        for (int32_t i = 0; i < I; ++i)
          acc += hval[i] * mx_element(down_codes[row * I + i], down_scales[row * ib + i / 32]);
        yt[o] += wj * acc;
      }
    }
  }
  free(xval);
  free(hval);
  return invalid;
}

/* ---------- Router (the input of the layer) --------------------------------
 * The tokens are routed to their top-k experts with renormalised softmax
 * weights ("Better MoE model inference with warp decode", Method: tokens are
 * routed to the top-k of E experts, e.g. top-8 of 128; sd114.wiki page,
 * 传统路径的困境). Per token: p = softmax(logits) over the E experts; the k
 * experts with the largest p, ties to the lower index, in descending order;
 * w_j = p_j / sum of the chosen p. Double precision throughout.
 */
int oracle_route(const float* logits, int32_t B, int32_t E, int32_t k, int32_t* ids,
                 double* w) {
  if (B < 0 || E <= 0 || k <= 0 || k > E) return -1;
  double* p = (double*)malloc(sizeof(double) * (size_t)E);
  unsigned char* taken = (unsigned char*)calloc((size_t)E, 1);
  if (!p || !taken) {
    free(p);
    free(taken);
    return -1;
  }
  for (int32_t b = 0; b < B; ++b) {
    const float* l = logits + (int64_t)b * E;
    double mx = -INFINITY;
    for (int32_t e = 0; e < E; ++e)
      if ((double)l[e] > mx) mx = (double)l[e];
    double z = 0.0;
    for (int32_t e = 0; e < E; ++e) {
      p[e] = exp((double)l[e] - mx);
      z += p[e];
    }
    for (int32_t e = 0; e < E; ++e) p[e] /= z;
    memset(taken, 0, (size_t)E);
    double sum = 0.0;
    for (int32_t j = 0; j < k; ++j) {
      int32_t best = -1;
      for (int32_t e = 0; e < E; ++e)
        if (!taken[e] && (best < 0 || p[e] > p[best])) best = e;
      taken[best] = 1;
      ids[(int64_t)b * k + j] = best;
      sum += p[best];
    }
    for (int32_t j = 0; j < k; ++j)
      w[(int64_t)b * k + j] = p[ids[(int64_t)b * k + j]] / sum;
  }
  free(p);
  free(taken);
  return 0;
}
