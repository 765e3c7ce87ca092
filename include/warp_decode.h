/*
 * warp_decode.h -- C ABI of the GB300-native output-centric ("warp decode")
 * MoE decode layer.
 *
 * The method ("Better MoE model inference with warp decode", TL;DR, Key claims
 * [§Reorganized parallelism] and [§How the two kernels work], Method; sd114.wiki
 * "Warp Decode" page, section 技术原理：两个 Kernel 搞定一切): for decode-time
 * MoE at small batch, give each warp one output scalar. The layer is two
 * kernels:
 *   moe_gate_up : one warp per (token, routed expert, intermediate neuron);
 *                 gate and up dot products share one read of the BF16
 *                 activation, MXFP8 weights are decoded exactly on the fly
 *                 and accumulated in FP32, SiLU(gate)*up is written as BF16.
 *   moe_down    : one warp per (token, output dim); one FP32 accumulator is
 *                 streamed over all top-k experts' down rows with the routing
 *                 weight folded in, then reduced across the 32 lanes by a
 *                 butterfly shuffle. No per-expert output buffer exists.
 * For batches where many routed pairs share each expert (see
 * LAYER KERNEL CHOICE below), the layer computes each step with an
 * expert-grouped kernel instead (moe_gate_up_grouped: one warp per (expert,
 * 8 neurons) for all the pairs routed to that expert; moe_down_grouped: one
 * CTA per 16 output rows for every token), multiplying on tensor cores and
 * decoding each weight once; each output is still written once, with the
 * same numerics up to FP32 rounding order.
 *
 * LAYER KERNEL CHOICE (moe_layer, moe_layer_noalloc, moe_layer_routed with
 * ids_out), with P = B * top_k routed pairs, measured on GB300 under uniform
 * routing:
 *   gate/up grouped when 8P >= 13E (H < 4096), 2P >= 3E (H >= 4096);
 *   down grouped when    4P >= 5E (I >= 3H), else 2P >= 5E (H < 6144),
 *                        P >= 2E (H >= 6144);
 * each only where the grouped kernel takes the shape and batch. The choice
 * is reported by moe_layer_gate_up_kernel and moe_layer_down_kernel.
 * moe_layer_host has the ids on the host and counts the batch's distinct
 * valid experts U instead (E <= 256):
 *   gate/up grouped when P >= 2 U (H < 4096), P >= 1.95 U (H >= 4096);
 *   down grouped when    P >= 1.5 U (I >= 3H), else P >= 2.6 U (H < 6144),
 *                        P >= 2.2 U (H >= 6144);
 * both only when 4P >= 3E or P >= 4U (below 3E/4 pairs, heavy sharing only);
 * the same break-even points under uniform routing, and earlier where the
 * pairs crowd onto few experts (skewed routing); moe_layer_host_kernels
 * reports that choice.
 *
 * Numerics (fixed by this API):
 *   g = sum_h x[t,h] Wg[e,n,h],  u = sum_h x[t,h] Wu[e,n,h]     (FP32 accum.)
 *   h[t,j,n] = bf16_rne( silu(g) * u ),  silu(g) = g / (1 + exp(-g))
 *   y[t,o]   = sum_j w[t,j] * sum_i h[t,j,i] Wd[e_j,o,i]          (FP32 accum.)
 * with MXFP8 weights (OCP MX v1.0): E4M3 codes, one E8M0 scale per 32
 * consecutive elements along the reduction axis (H for gate/up, I for down).
 *
 * Conventions for every entry point:
 *  - Shapes: H % 32 == 0 and H <= 8192, I % 32 == 0, E >= 1, top_k >= 1
 *    (ids may repeat, so top_k may exceed E, e.g. on a shard of the experts;
 *    routing from logits needs top_k <= E), B >= 0.
 *    B == 0 is a valid empty batch: nothing is launched, MOE_OK is returned.
 *  - Device pointers: caller-owned (e.g. torch allocations). The two code
 *    arrays (gu_codes, d_codes) must be 32-byte aligned, x and h 16-byte
 *    aligned, ids, w and y 4-byte aligned.
 *  - The library allocates no device memory, never synchronises, and enqueues
 *    its work on `stream` (a cudaStream_t; NULL = the legacy default stream).
 *  - Host-detectable problems (null pointer, bad shape, misalignment) return
 *    an error before anything is launched. A failed launch returns
 *    MOE_ERR_CUDA; moe_last_error() describes the last failure on this thread.
 *  - Expert ids are not checked on the host (that would need a copy back): a
 *    slot whose id is outside [0, E) contributes nothing, its intermediate is
 *    0, and if err_flag is non-NULL the device int32 *err_flag gets bit 0 set
 *    (it is never cleared by the library).
 *  - Duplicate ids in one token are allowed; their contributions add.
 *  - Device code has no traps, asserts or waits on flags.
 */
#ifndef WARP_DECODE_H
#define WARP_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_NULL = 1,        /* a required pointer is NULL */
  MOE_ERR_SHAPE = 2,       /* shape or batch outside the supported range */
  MOE_ERR_ALIGN = 3,       /* a pointer is not aligned as documented */
  MOE_ERR_CUDA = 4,        /* a CUDA call or kernel launch failed */
  MOE_ERR_UNSUPPORTED = 5  /* valid request this build does not implement */
} moe_status;

/* Layer shape: hidden size H, intermediate size I, E experts, top_k per token. */
typedef struct {
  int32_t H, I, E, top_k;
} moe_shape;

/*
 * Packed MXFP8 expert weights, device memory, written by moe_pack_weights:
 *   gu_codes  [E][I][2][H]    uint8 E4M3: for neuron n of expert e, the gate
 *                             row (H codes) followed by the up row (H codes),
 *                             so one warp streams one contiguous 2H-byte run.
 *   gu_scales [E][I][2][H/32] uint8 E8M0, same order (gate scales, up scales).
 *   d_codes   [E][H][I]       uint8 E4M3: down row o of expert e is contiguous.
 *   d_scales  [E][H][I/32]    uint8 E8M0.
 * Scale b of a row applies to elements 32b .. 32b+31 of that row.
 */
typedef struct {
  const uint8_t* gu_codes;
  const uint8_t* gu_scales;
  const uint8_t* d_codes;
  const uint8_t* d_scales;
} moe_weights;

/* Which packed array moe_packed_bytes sizes. */
enum { MOE_GU_CODES = 0, MOE_GU_SCALES = 1, MOE_D_CODES = 2, MOE_D_SCALES = 3 };

/* Bytes of packed array `which` for `shape` (all E experts); 0 if the shape
 * is invalid or `which` unknown. */
size_t moe_packed_bytes(const moe_shape* shape, int which);

/*
 * Quantise FP32 expert weights to MXFP8 and write the packed layout above.
 * Host memory in and out (runs on the CPU, no CUDA call). Inputs:
 *   w_gate [E][I][H], w_up [E][I][H], w_down [E][H][I]  (row-major FP32).
 * Rule (OCP MX v1.0 conversion): per 32-element block, shared exponent
 * floor(log2(max|v|)) - 8, stored as E8M0 (clamped to [0, 254]; an all-zero
 * block stores 0); elements v / 2^shared_exp rounded to nearest E4M3, ties to
 * even, magnitudes above 448 saturated to 448. Any `shape->E` works, so a
 * caller may pack one expert at a time (E = 1) into the matching offsets.
 */
moe_status moe_pack_weights(const moe_shape* shape, const float* w_gate, const float* w_up,
                            const float* w_down, uint8_t* gu_codes, uint8_t* gu_scales,
                            uint8_t* d_codes, uint8_t* d_scales);

/*
 * moe_gate_up -- first kernel ("moe_gate_up_3d_batched" on the pages).
 *   x    [B][H]        BF16 activations (device)
 *   ids  [B][top_k]    int32 expert ids (device)
 *   h    [B][top_k][I] BF16 intermediate, written (device)
 * h[t,j,n] = bf16_rne(silu(g)*u) for expert ids[t,j]; 0 for an invalid id.
 */
moe_status moe_gate_up(const moe_shape* shape, const moe_weights* w, const uint16_t* x,
                       const int32_t* ids, int32_t B, uint16_t* h, int32_t* err_flag,
                       void* stream);

/*
 * moe_gate_up_grouped -- moe_gate_up computed by its expert-grouped kernel:
 * one warp per (expert, 8 neurons) serves every (token, slot) pair routed to
 * that expert, decoding each weight once and multiplying on the tensor cores
 * (mma.sync m16n8k16, f16 operands, FP32 accumulation; rows are the gate and
 * up rows of the 8 neurons, columns 8 of the routed pairs). Each warp still
 * writes its own outputs h[t,j,n] once, with no buffer, gather or scatter
 * ("Better MoE model inference with warp decode", [§How the two kernels
 * work]; the routed experts of [§Reorganized parallelism]). Arguments and
 * result as for moe_gate_up; the sums differ from moe_gate_up's only in
 * FP32 rounding order (within each 32-element block, and the lower and the
 * upper half of H summed apart and then added); a pair's result does not
 * depend on the other pairs of the batch. Returns MOE_ERR_UNSUPPORTED, launching nothing, unless
 * H % 256 == 0, I % 64 == 0, E <= 256, gu_scales is 8-byte aligned and the
 * batch's pair lists fit in one CTA's shared memory.
 * moe_layer and the other layer entry points use this kernel by themselves
 * where the LAYER KERNEL CHOICE above says so (measured faster there on
 * GB300: each weight is decoded once instead of once per pair); elsewhere,
 * and when routing from logits without ids_out, they use moe_gate_up's
 * kernel. The two kernels agree to FP32 rounding order, so a token's result
 * can change in its last bits when the batch crosses the switch.
 */
moe_status moe_gate_up_grouped(const moe_shape* shape, const moe_weights* w,
                               const uint16_t* x, const int32_t* ids, int32_t B, uint16_t* h,
                               int32_t* err_flag, void* stream);

/*
 * moe_layer_gate_up_kernel -- which kernel the layer entry points (moe_layer,
 * moe_layer_noalloc, moe_layer_routed with ids_out; moe_layer_host decides
 * from its ids, see moe_layer_host_kernels) run for the gate/up step of a
 * batch of B tokens: *kernel_out = 0 for moe_gate_up's
 * per-token kernel, 1 for moe_gate_up_grouped's. A token's results can differ
 * in FP32 rounding order between the two, never beyond that. `w` may be NULL,
 * in which case gu_scales is taken to be suitably aligned; a non-NULL `w` has
 * its gate/up arrays checked as the layer entry points check them. Host-only
 * (no device call); returns MOE_ERR_SHAPE / MOE_ERR_NULL / MOE_ERR_ALIGN for a
 * bad shape, a NULL shape, kernel_out or gate/up array, or misaligned codes.
 */
moe_status moe_layer_gate_up_kernel(const moe_shape* shape, const moe_weights* w, int32_t B,
                                    int32_t* kernel_out);

/*
 * moe_down -- second kernel ("moe_down_3d_batched" on the pages).
 *   h    [B][top_k][I] BF16 intermediate from moe_gate_up (device)
 *   ids  [B][top_k]    int32 expert ids (device)
 *   wts  [B][top_k]    FP32 routing weights (device)
 *   y    [B][H]        FP32 output, overwritten (device)
 * y[t,o] = sum_j wts[t,j] * sum_i h[t,j,i] * Wd[ids[t,j], o, i].
 */
moe_status moe_down(const moe_shape* shape, const moe_weights* w, const uint16_t* h,
                    const int32_t* ids, const float* wts, int32_t B, float* y,
                    int32_t* err_flag, void* stream);

/*
 * moe_down_grouped -- moe_down computed by its expert-grouped kernel: one CTA
 * per 16 output rows o0..o0+15 serves every token of the batch. Its 12 warps
 * take the batch's routed experts in turn; for each, a warp streams rows
 * o0..o0+15 of that expert's down matrix once and multiplies them on the
 * tensor cores (mma.sync m16n8k16, f16 operands, FP32 accumulation; rows are
 * the 16 output dimensions, columns 8 of the pairs routed to the expert),
 * each block sum times its E8M0 scale, then adds routing weight x sum into
 * the warp's own partial sums of y in shared memory. The CTA adds its warps'
 * partial sums in a fixed order and writes every y[t,o] once: no atomics, no
 * per-expert output buffer, no combine in global memory ("Better MoE model
 * inference with warp decode", [§How the two kernels work], [§Buffer
 * elimination]); each down weight is decoded once per call instead of once
 * per (token, slot). Arguments and result as for moe_down; the sums differ
 * from moe_down's in FP32 rounding order, and a token's result can depend on
 * which other tokens share the batch in that order only. Results are the same
 * on every call with the same inputs. Returns MOE_ERR_UNSUPPORTED, launching
 * nothing, unless I % 256 == 0, E <= 256, 1 <= B <= 128 (B == 0 is an empty
 * batch), d_scales is 8-byte aligned and the batch's tables fit in one CTA's
 * shared memory. The layer entry points use this kernel by themselves where
 * the LAYER KERNEL CHOICE above says so and it takes the shape and batch.
 */
moe_status moe_down_grouped(const moe_shape* shape, const moe_weights* w, const uint16_t* h,
                            const int32_t* ids, const float* wts, int32_t B, float* y,
                            int32_t* err_flag, void* stream);

/*
 * moe_layer_down_kernel -- which kernel the layer entry points (moe_layer,
 * moe_layer_noalloc, moe_layer_routed with ids_out) run for the down step of
 * a batch of B tokens: *kernel_out = 0 for moe_down's
 * per-token kernel, 1 for moe_down_grouped's. Host-only; `w` may be NULL (the
 * scales are then taken to be aligned); errors as for moe_layer_gate_up_kernel,
 * with the down arrays of a non-NULL `w` checked.
 */
moe_status moe_layer_down_kernel(const moe_shape* shape, const moe_weights* w, int32_t B,
                                 int32_t* kernel_out);

/*
 * moe_layer_host_kernels -- the kernels moe_layer_host runs for a batch whose
 * ids_host [B][top_k] are given (host memory): *gate_up_out and *down_out =
 * 0 for the per-token kernel, 1 for the expert-grouped one (LAYER KERNEL
 * CHOICE above). Host-only; `w` may be NULL (scales taken to be aligned);
 * MOE_ERR_SHAPE for a bad shape, MOE_ERR_NULL for a NULL shape, output or
 * (B > 0) ids_host.
 */
moe_status moe_layer_host_kernels(const moe_shape* shape, const moe_weights* w,
                                  const int32_t* ids_host, int32_t B, int32_t* gate_up_out,
                                  int32_t* down_out);

/*
 * moe_layer -- the whole layer: the gate/up step then moe_down on `stream`.
 * Each step runs its per-token or its expert-grouped kernel as the LAYER
 * KERNEL CHOICE above says.
 * h_scratch [B][top_k][I] BF16 is caller-provided device memory that holds
 * the intermediate between the two kernels (its contents afterwards are the
 * intermediate, as from the gate/up kernel that ran).
 */
moe_status moe_layer(const moe_shape* shape, const moe_weights* w, const uint16_t* x,
                     const int32_t* ids, const float* wts, int32_t B, uint16_t* h_scratch,
                     float* y, int32_t* err_flag, void* stream);

/*
 * moe_layer_host -- the layer end to end from HOST buffers: copies x, ids and
 * wts host->device into the caller's device staging buffers (one
 * cudaMemcpyAsync each), runs the layer as moe_layer does with the kernels
 * chosen from ids_host (LAYER KERNEL CHOICE above), and copies y
 * device->host, all enqueued on `stream`. Returns once enqueued: synchronise
 * `stream` before reading y_host. Host buffers should be pinned for the
 * copies to be asynchronous. Shapes and device-buffer rules as for
 * moe_layer.
 */
moe_status moe_layer_host(const moe_shape* shape, const moe_weights* w, const uint16_t* x_host,
                          const int32_t* ids_host, const float* wts_host, int32_t B,
                          uint16_t* x_dev, int32_t* ids_dev, float* wts_dev, uint16_t* h_dev,
                          float* y_dev, float* y_host, int32_t* err_flag, void* stream);

/*
 * moe_route -- the router in front of the layer: for every token, the top_k
 * experts of softmax(logits) and their renormalised weights ("Better MoE
 * model inference with warp decode", Method: each token is routed to the
 * top-k of E experts, e.g. top-8 of 128).
 *   logits [B][E]     FP32 router logits (device), finite
 *   ids    [B][top_k] int32, written: experts by descending logit, ties to the
 *                     lower index
 *   wts    [B][top_k] FP32, written: exp(l_j - l_max) / sum over the chosen i
 *                     of exp(l_i - l_max) (= the softmax renormalised over the
 *                     chosen experts)
 * Needs E <= 256 and top_k <= min(32, E) (MOE_ERR_UNSUPPORTED otherwise).
 */
moe_status moe_route(const moe_shape* shape, const float* logits, int32_t B, int32_t* ids,
                     float* wts, void* stream);

/*
 * moe_layer_routed -- the layer from router logits (the same choice as
 * moe_route). Two ways, with the same results bit for bit where the layer
 * runs the per-token kernels (LAYER KERNEL CHOICE above):
 *  - ids_out and wts_out both non-NULL ([B][top_k], as moe_route): every token
 *    is routed once into them by the router kernel, and the layer reads that
 *    routing exactly as moe_layer does (same choice of gate/up kernel). The
 *    faster way.
 *  - both NULL: no ids/weights array exists at all. Every warp of moe_gate_up
 *    and moe_down routes its token from `logits` itself before it requests
 *    weights, which costs about 30 % of the layer at B=32. This way always
 *    uses the per-token kernels, so where the layer would run a grouped one
 *    it agrees with the other way to FP32 rounding order, not bit for bit.
 * Same limits as moe_route; other arguments as for moe_layer.
 */
moe_status moe_layer_routed(const moe_shape* shape, const moe_weights* w, const uint16_t* x,
                            const float* logits, int32_t B, uint16_t* h_scratch, float* y,
                            int32_t* ids_out, float* wts_out, int32_t* err_flag, void* stream);

/*
 * moe_layer_noalloc -- the whole layer (as moe_layer) for callers that cannot
 * allocate device memory: code that runs inside a host framework which owns
 * every device allocation through its own pool, or a latency-critical decode
 * loop that must not call cudaMalloc (it can synchronise the device). The
 * pages have no counterpart to this entry point.
 *   The intermediate lives in an array inside this library, of at most
 *   MOE_NOALLOC_MAX_INTERMEDIATE BF16 values (2 MiB) on every GPU that calls
 *   it, held until the library is unloaded. B * top_k * I above that limit
 *   returns MOE_ERR_SHAPE (moe_last_error() says why) before anything runs.
 *   The first call on each device looks up the array's device address with
 *   cudaGetSymbolAddress, with that device current; make that first call
 *   before any stream capture. The call allocates nothing. The address is
 *   kept for the rest of the process: after cudaDeviceReset on a device (which
 *   unloads this library's device code there, so the array may come back at
 *   another address) the kept address is stale, and this entry point must
 *   not be called on that device again.
 *   All calls share the one array: calls whose work overlaps on the GPU (for
 *   example on two streams at once) race on it. Each call overwrites every
 *   value it reads, so nothing needs clearing between calls.
 * Arguments, layouts and error behaviour otherwise as for moe_layer.
 */
#define MOE_NOALLOC_MAX_INTERMEDIATE (1u << 20)
moe_status moe_layer_noalloc(const moe_shape* shape, const moe_weights* w, const uint16_t* x,
                             const int32_t* ids, const float* wts, int32_t B, float* y,
                             int32_t* err_flag, void* stream);

/*
 * moe_local_ids -- expert parallelism (the layer split over G devices, each
 * holding a contiguous range of experts; y is then the sum of the devices'
 * results, one all-reduce). The slots of a batch that the shard holding
 * experts [e_first, e_first + e_count) computes:
 *   local_ids[t,j] = ids[t,j] - e_first  if e_first <= ids[t,j] < e_first + e_count
 *                    -1                  otherwise (contributes nothing on this shard)
 * A shard then runs the layer on its own experts (shape with E = e_count) with
 * local_ids and a NULL err_flag; ids outside [0, shape->E) (the global E) set
 * bit 0 of *err_flag here instead, if err_flag is non-NULL. ids and local_ids
 * [B][top_k] int32, device, 4-byte aligned. Requires 0 <= e_first and
 * 1 <= e_count <= shape->E - e_first (MOE_ERR_SHAPE otherwise). The pages
 * describe no multi-device split; this is the one the expert-major weight
 * layout allows with a single exchange.
 */
moe_status moe_local_ids(const moe_shape* shape, const int32_t* ids, int32_t B, int32_t e_first,
                         int32_t e_count, int32_t* local_ids, int32_t* err_flag, void* stream);

/* Static description of a status code. */
const char* moe_status_string(moe_status status);

/* Description of the last failure on the calling thread ("" if none). */
const char* moe_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* WARP_DECODE_H */
