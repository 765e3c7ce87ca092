/*
 * Seeded synthetic workload generator for the decode-time MoE layer.
 *
 * This file produces INPUTS only: activations, FP32 expert weights and the
 * router's (expert id, routing weight) pairs. It contains none of the layer's
 * arithmetic (no MXFP8 encoding or decoding, no dot products, no SwiGLU) and is
 * the single piece of code shared by the GPU path's benchmark/tests and the CPU
 * oracle's tests.
 *
 * Random numbers: a counter-based splitmix64 (Steele, Lea & Flood, "Fast
 * splittable pseudorandom number generators", OOPSLA 2014; constants as in
 * Vigna's public-domain splitmix64.c). The i-th output of a sequence whose
 * state starts at `key` is mix(key + (i+1)*golden), so any element of any
 * tensor can be drawn independently of the others (experts can be generated
 * one at a time, in parallel, in any order).
 * Normals: Box-Muller, cosine branch only, from outputs 2i and 2i+1.
 *
 * Workload shapes follow the "Qwen-3-style" MoE layer the pages benchmark
 * (top-8 of 128 experts, hidden 2048): see "Better MoE model inference with
 * warp decode", Key claims [§End-to-end decode throughput at scale] and
 * [§Buffer elimination].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define WL_GOLDEN 0x9E3779B97F4A7C15ULL

static uint64_t wl_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

/* i-th (0-based) output of the splitmix64 sequence whose state starts at key. */
uint64_t wl_splitmix64_at(uint64_t key, uint64_t i) {
  return wl_mix(key + (i + 1) * WL_GOLDEN);
}

/* Key of an independent stream: derived from (seed, stream id). */
uint64_t wl_stream_key(uint64_t seed, uint64_t stream) {
  return wl_splitmix64_at(wl_splitmix64_at(seed, stream), 0);
}

/* Uniform in [0,1) with 53 random bits. */
static double wl_uniform(uint64_t key, uint64_t i) {
  return (double)(wl_splitmix64_at(key, i) >> 11) * (1.0 / 9007199254740992.0);
}

/* Standard normal number i of stream `key` (Box-Muller, cosine branch). */
double wl_normal_at(uint64_t key, uint64_t i) {
  const double two_pi = 6.283185307179586476925286766559;
  double u1 = wl_uniform(key, 2 * i);
  double u2 = wl_uniform(key, 2 * i + 1);
  double r = sqrt(-2.0 * log(1.0 - u1)); /* 1-u1 in (0,1]: log finite */
  return r * cos(two_pi * u2);
}

/* out[i] = (float)(mean + std * normal(key, start + i)), i < count. */
void wl_normal_f32(uint64_t key, uint64_t start, uint64_t count, double mean,
                   double std, float* out) {
  for (uint64_t i = 0; i < count; ++i)
    out[i] = (float)(mean + std * wl_normal_at(key, start + i));
}

/* float -> bfloat16 bits, round to nearest even (inputs are finite). */
static uint16_t wl_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

/* BF16 activations: N(0,1) drawn in double, rounded to float, then to bf16. */
void wl_normal_bf16(uint64_t key, uint64_t start, uint64_t count, uint16_t* out) {
  for (uint64_t i = 0; i < count; ++i)
    out[i] = wl_f32_to_bf16((float)wl_normal_at(key, start + i));
}

/*
 * Router stand-in (the router is an input to the layer, not part of it):
 *   logits[b,e] = normal(logit_key, b*E + e) + bias_std * normal(bias_key, e)
 *   p = softmax(logits[b,:]); take the top_k largest p (ties: lower expert
 *   index first), renormalise the chosen p to sum 1.
 * ids[b*top_k + j] and weights[b*top_k + j] are written in descending-p order.
 * Returns 0, or -1 on bad arguments.
 */
int wl_route(uint64_t logit_key, uint64_t bias_key, double bias_std, int32_t B,
             int32_t E, int32_t top_k, int32_t* ids, float* weights) {
  if (B < 0 || E <= 0 || top_k <= 0 || top_k > E) return -1;
  double* p = (double*)malloc(sizeof(double) * (size_t)E);
  unsigned char* taken = (unsigned char*)malloc((size_t)E);
  if (!p || !taken) {
    free(p);
    free(taken);
    return -1;
  }
  for (int32_t b = 0; b < B; ++b) {
    double mx = -INFINITY;
    for (int32_t e = 0; e < E; ++e) {
      double l = wl_normal_at(logit_key, (uint64_t)b * (uint64_t)E + (uint64_t)e);
      if (bias_std != 0.0) l += bias_std * wl_normal_at(bias_key, (uint64_t)e);
      p[e] = l;
      if (l > mx) mx = l;
    }
    double z = 0.0;
    for (int32_t e = 0; e < E; ++e) {
      p[e] = exp(p[e] - mx);
      z += p[e];
    }
    for (int32_t e = 0; e < E; ++e) p[e] /= z;
    memset(taken, 0, (size_t)E);
    double chosen_sum = 0.0;
    for (int32_t j = 0; j < top_k; ++j) {
      int32_t best = -1;
      for (int32_t e = 0; e < E; ++e)
        if (!taken[e] && (best < 0 || p[e] > p[best])) best = e;
      taken[best] = 1;
      ids[b * top_k + j] = best;
      chosen_sum += p[best];
    }
    for (int32_t j = 0; j < top_k; ++j)
      weights[b * top_k + j] = (float)(p[ids[b * top_k + j]] / chosen_sum);
  }
  free(p);
  free(taken);
  return 0;
}

/* The router logits wl_route draws, as FP32 [B][E] (for a router run by the
 * caller): logits[b,e] = (float)(normal(logit_key, b*E + e)
 *                                + bias_std * normal(bias_key, e)). */
void wl_logits(uint64_t logit_key, uint64_t bias_key, double bias_std, int32_t B, int32_t E,
               float* out) {
  for (int32_t b = 0; b < B; ++b)
    for (int32_t e = 0; e < E; ++e) {
      double l = wl_normal_at(logit_key, (uint64_t)b * (uint64_t)E + (uint64_t)e);
      if (bias_std != 0.0) l += bias_std * wl_normal_at(bias_key, (uint64_t)e);
      out[(size_t)b * E + e] = (float)l;
    }
}
