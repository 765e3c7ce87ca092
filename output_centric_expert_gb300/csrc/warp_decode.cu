// C-ABI entry points of the output-centric ("warp decode") MoE decode layer:
// argument checks, the composition of the two kernels into a layer, the
// router kernel and the allocation-free layer variant. The kernels themselves
// are in wd_gate_up.cu and wd_down.cu, their shared device code in
// wd_device.cuh.
#include <mutex>

#include "wd_device.cuh"
#include "wd_down_grouped.h"
#include "wd_gate_up_grouped.h"

namespace wd {

thread_local char g_last_error[256] = "";

void set_error(const char* what, cudaError_t e) {
  snprintf(g_last_error, sizeof(g_last_error), "%s: %s", what, cudaGetErrorString(e));
}

void set_error_msg(const char* msg) { snprintf(g_last_error, sizeof(g_last_error), "%s", msg); }

int sm_count() {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static int cached[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 152;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 152;
    cached[dev] = n;
  }
  return cached[dev];
}

namespace {

// moe_local_ids: one thread per (token, slot).
__global__ void __launch_bounds__(kThreads)
    moe_local_ids_kernel(const int32_t* __restrict__ ids, int32_t* __restrict__ local, int P,
                         int E, int e_first, int e_count, int32_t* __restrict__ err) {
  const int p = blockIdx.x * kThreads + threadIdx.x;
  if (p >= P) return;
  const int e = __ldg(ids + p);
  if (e < 0 || e >= E) flag_invalid(err);
  local[p] = (e >= e_first && e < e_first + e_count) ? e - e_first : -1;
}

// moe_route: one warp per token.
__global__ void __launch_bounds__(kThreads)
    moe_route_kernel(const float* __restrict__ logits, int32_t* __restrict__ ids,
                     float* __restrict__ wts, int B, int E, int top_k) {
  launch_dependents();  // moe_layer_routed's gate/up kernel waits for the ids itself
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


moe_status check_shape(const moe_shape* s, int32_t B) {
  if (!s) return MOE_ERR_NULL;
  if (s->H <= 0 || s->I <= 0 || s->E <= 0 || s->top_k <= 0 || B < 0 || s->H % 32 || s->I % 32) {
    set_error_msg("shape: need H%32==0, I%32==0, E>=1, top_k>=1, B>=0");
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

moe_status launch_status(const char* what) {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error(what, e);
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

// Checks of the routed entry points: the warp router handles E <= 256 and
// top_k <= 32 distinct choices (top_k <= E); logits are FP32 [B][E], 4-byte
// aligned.
moe_status check_route(const moe_shape* s, const float* logits) {
  if (!logits) return MOE_ERR_NULL;
  if (s->E > kRouteMaxE || s->top_k > 32 || s->top_k > s->E) {
    set_error_msg("routing on the device needs E <= 256 and top_k <= min(32, E)");
    return MOE_ERR_UNSUPPORTED;
  }
  if (!aligned(logits, 4)) {
    set_error_msg("alignment: logits need 4 bytes");
    return MOE_ERR_ALIGN;
  }
  return MOE_OK;
}

// Which kernel computes the intermediate: the per-token one of moe_gate_up
// (slots per warp chosen by the batch) or the expert-grouped one.
enum class GateUpForm { kPerToken, kGrouped };

moe_status gate_up_impl(const moe_shape* s, const moe_weights* w, const uint16_t* x,
                        const int32_t* ids, int32_t B, uint16_t* h, int32_t* err,
                        cudaStream_t st, RouteArgs route = kNoRoute,
                        GateUpForm form = GateUpForm::kPerToken) {
  moe_status rc = check_shape(s, B);
  if (rc != MOE_OK) return rc;
  if ((rc = check_weights(w, true, false)) != MOE_OK) return rc;
  if (form == GateUpForm::kGrouped && !gate_up_grouped_supported(s, w, B)) {
    set_error_msg("moe_gate_up_grouped: needs H % 256 == 0, I % 64 == 0, E <= 256, 8-byte "
                  "aligned gu_scales and the batch's tables within shared memory");
    return MOE_ERR_UNSUPPORTED;
  }
  if (B == 0) return MOE_OK;
  if (!x || (!ids && !route.logits) || !h) return MOE_ERR_NULL;
  if (!aligned(x, 16) || !aligned(h, 16) || !aligned(ids, 4) || !aligned(err, 4)) {
    set_error_msg("alignment: x and h need 16 bytes, ids and err_flag 4");
    return MOE_ERR_ALIGN;
  }
  if (form == GateUpForm::kGrouped)
    rc = launch_gate_up_grouped(s, w, x, ids, B, h, err, st, route.dependent);
  else
    rc = launch_gate_up_kernels(s, w, x, ids, B, h, err, st, route);
  if (rc != MOE_OK) return rc;
  return launch_status("moe_gate_up launch");
}

// The form of moe_gate_up a layer entry point uses: the expert-grouped kernel
// once the batch has enough pairs per expert, if the shape allows it. The
// switch points are measured on GB300 in the layer (CUDA graph, cold L2,
// uniform routing, the down step per-token): per-token vs grouped gate/up
// break even at about 25 tokens for the Qwen-3-30B-A3B shape (1.56 E pairs;
// H = 2048: 24 tokens 95.2 us per-token vs 97.1 with the grouped gate/up, 26
// tokens 101.1 vs 100.7, 28 tokens 104.5 vs 101.7), 24 for the
// Qwen-3-235B-A22B shape (1.5 E; H = 4096: 22 tokens 331.0 vs 337.7, 24
// tokens 356.2 vs 357.1, 26 tokens 390.3 vs 357.2), 6 for the Mixtral shape
// (1.5 E; 5 tokens 221.4 vs 230.7, 6 tokens 259.4 vs 255.4) and 48 for the
// DeepSeek-V3 shape (1.5 E; H = 7168: 44 tokens 1536.6 vs 1584.6, 48 tokens
// 1653.4 vs 1659.8, 52 tokens 1985.0 vs 1728.5).
GateUpForm layer_form(const moe_shape* s, const moe_weights* w, int32_t B) {
  if (!s) return GateUpForm::kPerToken;
  const int64_t pairs = (int64_t)B * s->top_k, E = s->E;
  const bool shared = s->H >= 4096 ? 2 * pairs >= 3 * E    // 1.5 E pairs
                                   : 8 * pairs >= 13 * E;  // 1.625 E
  if (shared && gate_up_grouped_supported(s, w, B)) return GateUpForm::kGrouped;
  return GateUpForm::kPerToken;
}

// Which kernel computes y: the per-token one of moe_down (outputs per warp
// chosen by the batch) or the expert-grouped one.
enum class DownForm { kPerToken, kGrouped };

moe_status down_impl(const moe_shape* s, const moe_weights* w, const uint16_t* h,
                     const int32_t* ids, const float* wts, int32_t B, float* y, int32_t* err,
                     cudaStream_t st, bool dependent, const float* logits = nullptr,
                     DownForm form = DownForm::kPerToken) {
  moe_status rc = check_shape(s, B);
  if (rc != MOE_OK) return rc;
  if ((rc = check_weights(w, false, true)) != MOE_OK) return rc;
  if (form == DownForm::kGrouped && B > 0 && !down_grouped_supported(s, w, B)) {
    set_error_msg("moe_down_grouped: needs I % 256 == 0, E <= 256, B <= 128, 8-byte aligned "
                  "d_scales and the batch's tables within shared memory");
    return MOE_ERR_UNSUPPORTED;
  }
  if (B == 0) return MOE_OK;
  if (!h || ((!ids || !wts) && !logits) || !y) return MOE_ERR_NULL;
  if (!aligned(h, 16) || !aligned(ids, 4) || !aligned(wts, 4) || !aligned(y, 4) ||
      !aligned(err, 4)) {
    set_error_msg("alignment: h needs 16 bytes, ids/wts/y/err_flag 4");
    return MOE_ERR_ALIGN;
  }
  if (form == DownForm::kGrouped)
    rc = launch_down_grouped(s, w, h, ids, wts, B, y, err, st, dependent);
  else
    rc = launch_down_kernels(s, w, h, ids, wts, B, y, err, st, dependent, logits);
  if (rc != MOE_OK) return rc;
  return launch_status("moe_down launch");
}

// The form of moe_down a layer entry point uses: the expert-grouped kernel once
// the batch has enough pairs per expert, if it takes the shape and batch.
// Measured on GB300 (each kernel alone, CUDA graph, cold L2, uniform
// routing), per-token vs grouped down break even at about 37 tokens for the
// Qwen-3-30B-A3B shape (43.8 vs 46.4 us at 32, 52.2 vs 50.7 at 40), 33 for
// the Qwen-3-235B-A22B shape and 55 for the DeepSeek-V3 shape (1.7 E). Rows
// of the intermediate much longer than the output (I >= 3H: the Mixtral
// shape's 14336 against 4096) make each token's down rows long for the
// per-token kernel: there the grouped down wins from 1.25 E pairs (layer with
// the per-token gate/up: 4 tokens 170.7 us per-token down vs 172.3 grouped,
// 5 tokens 221.4 vs 204.3).
DownForm layer_down_form(const moe_shape* s, const moe_weights* w, int32_t B) {
  if (!s) return DownForm::kPerToken;
  const int64_t pairs = (int64_t)B * s->top_k, E = s->E;
  const bool shared = s->I >= 3 * (int64_t)s->H ? 4 * pairs >= 5 * E
                      : s->H >= 6144           ? pairs >= 2 * E
                                               : 2 * pairs >= 5 * E;
  if (shared && down_grouped_supported(s, w, B)) return DownForm::kGrouped;
  return DownForm::kPerToken;
}

// The forms for a batch whose ids are on the host: the same measured
// break-even points written as pairs per used expert, P >= tau * U with U the
// distinct experts of the batch, so that a batch whose pairs crowd onto few
// experts (skewed routing) takes the grouped kernels where they win. With
// uniform routing U = E (1 - (1 - k/E)^B) on average, and the thresholds
// reproduce the rules on P and E at the measured shapes: gate/up tau = 2.0
// (H < 4096; Qwen-3-30B-A3B: 1.98 pairs per used expert at 24 tokens, 2.05
// at 26) or 1.95 (H >= 4096; Qwen-3-235B-A22B 1.94 at 23 tokens and 1.98 at
// 24, DeepSeek-V3 shape 1.92 at 48); down tau = 2.6 (H < 6144), 2.2 (H >=
// 6144; DeepSeek-V3 shape 2.1 at 55 tokens) or 1.5 (I >= 3H; Mixtral shape
// 1.46 at 4 tokens, 1.64 at 5). Below 3E/4 pairs the grouped kernels' fixed
// costs (every CTA lists the pairs, stages activations) need more sharing
// than that: they are taken there only from 4 pairs per used expert
// (Qwen-3-30B-A3B skewed batches: 8 tokens, 64 pairs, 2.4 per used expert,
// layer 34.7 us per-token vs 36.5 with the grouped gate/up; 12 tokens, 96
// pairs, 45.8 us both grouped vs 50.3). Skewed Qwen-3-30B-A3B batch of 32
// tokens (43 used experts, 6 pairs each): gate/up 40.6 us grouped against
// 73.8 per-token, down 34.9 against 38.4.
struct LayerForms {
  GateUpForm gate_up;
  DownForm down;
};

LayerForms layer_forms_for_ids(const moe_shape* s, const moe_weights* w, const int32_t* ids,
                               int32_t B) {
  LayerForms f = {GateUpForm::kPerToken, DownForm::kPerToken};
  if (s->E > kRouteMaxE) return f;  // beyond the grouped kernels' expert count
  uint64_t used[kRouteMaxE / 64] = {};
  const int64_t P = (int64_t)B * s->top_k;
  int64_t U = 0;
  for (int64_t p = 0; p < P; ++p) {
    const int32_t e = ids[p];
    if (e < 0 || e >= s->E) continue;
    const uint64_t bit = 1ull << (e & 63);
    if (!(used[e >> 6] & bit)) {
      used[e >> 6] |= bit;
      ++U;
    }
  }
  if (U == 0) return f;
  const bool enough = 4 * P >= 3 * (int64_t)s->E || P >= 4 * U;
  const bool gu_shared = enough && (s->H >= 4096 ? 20 * P >= 39 * U : P >= 2 * U);
  const bool dn_shared = enough && (s->I >= 3 * (int64_t)s->H ? 2 * P >= 3 * U
                                    : s->H >= 6144           ? 5 * P >= 11 * U
                                                             : 5 * P >= 13 * U);
  if (gu_shared && gate_up_grouped_supported(s, w, B)) f.gate_up = GateUpForm::kGrouped;
  if (dn_shared && down_grouped_supported(s, w, B)) f.down = DownForm::kGrouped;
  return f;
}

// The layer with the given forms (arguments validated by the caller): the
// down kernel is launched as a programmatic dependent of the gate/up kernel.
moe_status layer_run(const moe_shape* s, const moe_weights* w, const uint16_t* x,
                     const int32_t* ids, const float* wts, int32_t B, uint16_t* h, float* y,
                     int32_t* err, cudaStream_t st, LayerForms f) {
  moe_status rc = gate_up_impl(s, w, x, ids, B, h, err, st, kNoRoute, f.gate_up);
  if (rc != MOE_OK) return rc;
  return down_impl(s, w, h, ids, wts, B, y, err, st, true, nullptr, f.down);
}

}  // namespace
}  // namespace wd

extern "C" moe_status moe_gate_up(const moe_shape* shape, const moe_weights* w,
                                  const uint16_t* x, const int32_t* ids, int32_t B,
                                  uint16_t* h, int32_t* err_flag, void* stream) {
  using namespace wd;
  return gate_up_impl(shape, w, x, ids, B, h, err_flag, (cudaStream_t)stream);
}

extern "C" moe_status moe_gate_up_grouped(const moe_shape* shape, const moe_weights* w,
                                          const uint16_t* x, const int32_t* ids, int32_t B,
                                          uint16_t* h, int32_t* err_flag, void* stream) {
  using namespace wd;
  return gate_up_impl(shape, w, x, ids, B, h, err_flag, (cudaStream_t)stream, kNoRoute,
                      GateUpForm::kGrouped);
}

extern "C" moe_status moe_layer_gate_up_kernel(const moe_shape* shape, const moe_weights* w,
                                               int32_t B, int32_t* kernel_out) {
  using namespace wd;
  if (!kernel_out) return MOE_ERR_NULL;
  moe_status rc = check_shape(shape, B);
  if (rc != MOE_OK) return rc;
  if (w && (rc = check_weights(w, true, false)) != MOE_OK) return rc;
  *kernel_out = layer_form(shape, w, B) == GateUpForm::kGrouped ? 1 : 0;
  return MOE_OK;
}

extern "C" moe_status moe_down(const moe_shape* shape, const moe_weights* w, const uint16_t* h,
                               const int32_t* ids, const float* wts, int32_t B, float* y,
                               int32_t* err_flag, void* stream) {
  using namespace wd;
  return down_impl(shape, w, h, ids, wts, B, y, err_flag, (cudaStream_t)stream, false);
}

extern "C" moe_status moe_down_grouped(const moe_shape* shape, const moe_weights* w,
                                       const uint16_t* h, const int32_t* ids, const float* wts,
                                       int32_t B, float* y, int32_t* err_flag, void* stream) {
  using namespace wd;
  return down_impl(shape, w, h, ids, wts, B, y, err_flag, (cudaStream_t)stream, false, nullptr,
                   DownForm::kGrouped);
}

extern "C" moe_status moe_layer_down_kernel(const moe_shape* shape, const moe_weights* w,
                                            int32_t B, int32_t* kernel_out) {
  using namespace wd;
  if (!kernel_out) return MOE_ERR_NULL;
  moe_status rc = check_shape(shape, B);
  if (rc != MOE_OK) return rc;
  if (w && (rc = check_weights(w, false, true)) != MOE_OK) return rc;
  *kernel_out = layer_down_form(shape, w, B) == DownForm::kGrouped ? 1 : 0;
  return MOE_OK;
}

extern "C" moe_status moe_layer_host_kernels(const moe_shape* shape, const moe_weights* w,
                                             const int32_t* ids_host, int32_t B,
                                             int32_t* gate_up_out, int32_t* down_out) {
  using namespace wd;
  if (!gate_up_out || !down_out) return MOE_ERR_NULL;
  moe_status rc = check_shape(shape, B);
  if (rc != MOE_OK) return rc;
  if (w && (rc = check_weights(w, true, true)) != MOE_OK) return rc;
  if (B > 0 && !ids_host) return MOE_ERR_NULL;
  const LayerForms f = B > 0 ? layer_forms_for_ids(shape, w, ids_host, B)
                             : LayerForms{GateUpForm::kPerToken, DownForm::kPerToken};
  *gate_up_out = f.gate_up == GateUpForm::kGrouped ? 1 : 0;
  *down_out = f.down == DownForm::kGrouped ? 1 : 0;
  return MOE_OK;
}

extern "C" moe_status moe_layer(const moe_shape* shape, const moe_weights* w, const uint16_t* x,
                                const int32_t* ids, const float* wts, int32_t B,
                                uint16_t* h_scratch, float* y, int32_t* err_flag,
                                void* stream) {
  using namespace wd;
  // validate everything before the first launch, so a bad argument launches nothing
  moe_status rc = check_shape(shape, B);
  if (rc != MOE_OK) return rc;
  if ((rc = check_weights(w, true, true)) != MOE_OK) return rc;
  if (B == 0) return MOE_OK;
  if (!x || !ids || !wts || !h_scratch || !y) return MOE_ERR_NULL;
  return layer_run(shape, w, x, ids, wts, B, h_scratch, y, err_flag, (cudaStream_t)stream,
                   {layer_form(shape, w, B), layer_down_form(shape, w, B)});
}

extern "C" moe_status moe_route(const moe_shape* shape, const float* logits, int32_t B,
                                int32_t* ids, float* wts, void* stream) {
  using namespace wd;
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
  using namespace wd;
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
  cudaStream_t st = (cudaStream_t)stream;
  if (ids_out) {
    // The routing has a home: route every token once into it, then run the
    // layer on it (Q30 B=32: 112.1 us, moe_layer on the same ids 108.6, against
    // 161.2 us when every CTA of both kernels routes its token itself before it
    // can request any weights).
    const unsigned grid = (unsigned)((B + kWarpsPerCta - 1) / kWarpsPerCta);
    moe_route_kernel<<<grid, kThreads, 0, st>>>(logits, ids_out, wts_out, B, shape->E,
                                                 shape->top_k);
    if ((rc = launch_status("moe_route launch")) != MOE_OK) return rc;
    // the gate/up kernel is a programmatic dependent of the router: its CTAs
    // are resident when the ids are written (B=1 16.1 -> 15.8 us, B=32 113.6 ->
    // 112.1). It releases moe_down, which reads the ids before its own wait,
    // only after its wait for the router.
    const RouteArgs after_router = {nullptr, true};
    rc = gate_up_impl(shape, w, x, ids_out, B, h_scratch, err_flag, st, after_router,
                      layer_form(shape, w, B));
    if (rc != MOE_OK) return rc;
    return down_impl(shape, w, h_scratch, ids_out, wts_out, B, y, err_flag, st, true, nullptr,
                     layer_down_form(shape, w, B));
  }
  const RouteArgs route = {logits, false};
  rc = gate_up_impl(shape, w, x, nullptr, B, h_scratch, err_flag, st, route);
  if (rc != MOE_OK) return rc;
  return down_impl(shape, w, h_scratch, nullptr, nullptr, B, y, err_flag, st, true, logits);
}

extern "C" moe_status moe_layer_host(const moe_shape* shape, const moe_weights* w,
                                     const uint16_t* x_host, const int32_t* ids_host,
                                     const float* wts_host, int32_t B, uint16_t* x_dev,
                                     int32_t* ids_dev, float* wts_dev, uint16_t* h_dev,
                                     float* y_dev, float* y_host, int32_t* err_flag,
                                     void* stream) {
  using namespace wd;
  moe_status rc = check_shape(shape, B);
  if (rc != MOE_OK) return rc;
  if ((rc = check_weights(w, true, true)) != MOE_OK) return rc;
  if (B == 0) return MOE_OK;
  if (!x_host || !ids_host || !wts_host || !y_host || !x_dev || !ids_dev || !wts_dev || !h_dev ||
      !y_dev)
    return MOE_ERR_NULL;
  if (!aligned(x_dev, 16) || !aligned(h_dev, 16) || !aligned(ids_dev, 4) ||
      !aligned(wts_dev, 4) || !aligned(y_dev, 4) || !aligned(err_flag, 4)) {
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
  // the ids are on the host: the kernels are chosen from the batch's own
  // pairs per used expert
  rc = layer_run(shape, w, x_dev, ids_dev, wts_dev, B, h_dev, y_dev, err_flag, st,
                 layer_forms_for_ids(shape, w, ids_host, B));
  if (rc != MOE_OK) return rc;
  if ((e = cudaMemcpyAsync(y_host, y_dev, nx * 4, cudaMemcpyDeviceToHost, st)) != cudaSuccess) {
    set_error("moe_layer_host: device->host copy", e);
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

extern "C" moe_status moe_local_ids(const moe_shape* shape, const int32_t* ids, int32_t B,
                                    int32_t e_first, int32_t e_count, int32_t* local_ids,
                                    int32_t* err_flag, void* stream) {
  using namespace wd;
  moe_status rc = check_shape(shape, B);
  if (rc != MOE_OK) return rc;
  if (e_first < 0 || e_count < 1 || e_count > shape->E - e_first) {
    set_error_msg("moe_local_ids: need 0 <= e_first and 1 <= e_count <= E - e_first");
    return MOE_ERR_SHAPE;
  }
  if (B == 0) return MOE_OK;
  if (!ids || !local_ids) return MOE_ERR_NULL;
  if (!aligned(ids, 4) || !aligned(local_ids, 4) || !aligned(err_flag, 4)) {
    set_error_msg("alignment: ids, local_ids and err_flag need 4 bytes");
    return MOE_ERR_ALIGN;
  }
  const int64_t P = (int64_t)B * shape->top_k;
  const unsigned grid = (unsigned)((P + kThreads - 1) / kThreads);
  moe_local_ids_kernel<<<grid, kThreads, 0, (cudaStream_t)stream>>>(
      ids, local_ids, (int)P, shape->E, e_first, e_count, err_flag);
  return launch_status("moe_local_ids launch");
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

extern "C" const char* moe_last_error(void) { return wd::g_last_error; }

// ------------------------------------------ allocation-free layer variant --
// moe_layer_noalloc: the whole layer with the intermediate kept in a fixed
// array that belongs to this library instead of a caller-provided buffer, for
// callers that cannot allocate device memory themselves. The array lives for
// as long as the library is loaded, on every GPU that uses it.

static __device__ __align__(256) uint16_t g_noalloc_intermediate[MOE_NOALLOC_MAX_INTERMEDIATE];

namespace wd {
namespace {

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mutex;
uint16_t* g_noalloc_ptr[kNoAllocMaxDevices] = {};

// Device address of the fixed intermediate array on the current device. Host
// code must not pass the array's name to a kernel (on the host it only stands
// for the symbol), so the address is looked up once per device, with that
// device current, and cached for the rest of the process (a cudaDeviceReset
// makes the cached address stale; the header says so).
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
}  // namespace wd

extern "C" moe_status moe_layer_noalloc(const moe_shape* shape, const moe_weights* w,
                                        const uint16_t* x, const int32_t* ids, const float* wts,
                                        int32_t B, float* y, int32_t* err_flag, void* stream) {
  using namespace wd;
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
  rc = gate_up_impl(shape, w, x, ids, B, h, err_flag, (cudaStream_t)stream, kNoRoute,
                    layer_form(shape, w, B));
  if (rc != MOE_OK) return rc;
  return down_impl(shape, w, h, ids, wts, B, y, err_flag, (cudaStream_t)stream, true, nullptr,
                   layer_down_form(shape, w, B));
}
