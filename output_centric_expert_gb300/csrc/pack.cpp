// Host-side MXFP8 packer: FP32 expert weights -> the packed layout the two
// kernels stream (see include/warp_decode.h for the layout).
//
// The pages only name the weight format "MXFP8" with an on-the-fly upcast
// ("Better MoE model inference with warp decode", Key claims
// [§How the two kernels work]); element and scale types follow OCP MX v1.0:
// E4M3 elements, one E8M0 scale per 32 consecutive elements of a row.
#include <algorithm>
#include <cfenv>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "warp_decode.h"

namespace {

// E8M0 scale code of one 32-element block: shared exponent
// floor(log2(amax)) - 8 (8 = exponent of E4M3's largest normal), biased by
// 127 and clamped to the finite E8M0 range; an all-zero block gets code 0.
uint8_t block_scale_code(const float* v) {
  float amax = 0.0f;
  for (int i = 0; i < 32; ++i) amax = std::max(amax, std::fabs(v[i]));
  if (amax == 0.0f) return 0;
  if (std::isinf(amax)) return 254;
  int e2;
  std::frexp(amax, &e2);  // amax = f * 2^e2, f in [0.5, 1)
  int code = (e2 - 1) - 8 + 127;
  return (uint8_t)std::min(254, std::max(0, code));
}

// Nearest E4M3 code (ties to even) of a value already divided by its block
// scale; magnitudes beyond 448 saturate to 448.
uint8_t e4m3_rne(double v) {
  if (std::isnan(v)) return 0x7F;
  const uint8_t sign = std::signbit(v) ? 0x80 : 0x00;
  const double a = std::fabs(v);
  if (a >= 448.0) return sign | 0x7E;
  int e2;
  std::frexp(a, &e2);
  const int ex = std::max(e2 - 1, -6);  // subnormals share exponent -6's quantum
  const double q = std::nearbyint(std::ldexp(a, 3 - ex));  // units of 2^(ex-3)
  int code;
  if (q < 8.0)
    code = (int)q;  // subnormal (only reachable with ex == -6)
  else if (q >= 16.0)
    code = (ex + 8) << 3;  // rounded up into the next binade
  else
    code = ((ex + 7) << 3) | ((int)q - 8);
  return sign | (uint8_t)std::min(code, 0x7E);
}

// Quantise one row of K values into codes and K/32 scales.
void pack_row(const float* src, int64_t K, uint8_t* codes, uint8_t* scales) {
  for (int64_t b = 0; b < K / 32; ++b) {
    const float* v = src + b * 32;
    const uint8_t s = block_scale_code(v);
    scales[b] = s;
    for (int i = 0; i < 32; ++i)
      codes[b * 32 + i] = e4m3_rne(std::ldexp((double)v[i], 127 - (int)s));
  }
}

bool shape_ok(const moe_shape* s) {
  return s && s->H > 0 && s->I > 0 && s->E > 0 && s->top_k > 0 &&
         s->H % 32 == 0 && s->I % 32 == 0;
}

}  // namespace

extern "C" size_t moe_packed_bytes(const moe_shape* s, int which) {
  if (!shape_ok(s)) return 0;
  const size_t E = (size_t)s->E, H = (size_t)s->H, I = (size_t)s->I;
  switch (which) {
    case MOE_GU_CODES: return E * I * 2 * H;
    case MOE_GU_SCALES: return E * I * 2 * (H / 32);
    case MOE_D_CODES: return E * H * I;
    case MOE_D_SCALES: return E * H * (I / 32);
    default: return 0;
  }
}

extern "C" moe_status moe_pack_weights(const moe_shape* s, const float* w_gate,
                                       const float* w_up, const float* w_down,
                                       uint8_t* gu_codes, uint8_t* gu_scales,
                                       uint8_t* d_codes, uint8_t* d_scales) {
  if (!s || !w_gate || !w_up || !w_down || !gu_codes || !gu_scales || !d_codes || !d_scales)
    return MOE_ERR_NULL;
  if (!shape_ok(s)) return MOE_ERR_SHAPE;
  const int old_round = std::fegetround();
  std::fesetround(FE_TONEAREST);
  const int64_t E = s->E, H = s->H, I = s->I;
  for (int64_t e = 0; e < E; ++e) {
    for (int64_t n = 0; n < I; ++n) {
      const int64_t src = (e * I + n) * H;
      const int64_t dst = (e * I + n) * 2;  // [gate, up] rows of neuron n
      pack_row(w_gate + src, H, gu_codes + dst * H, gu_scales + dst * (H / 32));
      pack_row(w_up + src, H, gu_codes + (dst + 1) * H, gu_scales + (dst + 1) * (H / 32));
    }
    for (int64_t o = 0; o < H; ++o) {
      const int64_t r = e * H + o;
      pack_row(w_down + r * I, I, d_codes + r * I, d_scales + r * (I / 32));
    }
  }
  std::fesetround(old_round);
  return MOE_OK;
}
