"""Accuracy study of the method's claim, on the CPU oracle.

"Better MoE model inference with warp decode", Key claims [§Improved accuracy]:
activations stay BF16 and accumulators FP32, so the conventional path's
BF16 -> MXFP8 -> BF16 activation round trip is skipped, and the outputs come
out closer to a full-precision reference. The pages do not define that
reference, so two readings are measured:

* the same MXFP8 weights with exact (unrounded) activations, in FP64;
* the unquantised FP32 weights with exact activations, in FP64.

The first tests pin oracle.moe_layer_variant against torch (float8 casts,
float64 matmuls); the study test then reports the error ratio on synthetic
Qwen-3-30B-shaped inputs and checks its direction.
"""
import numpy as np
import pytest
import torch

import oracle
from output_centric_expert_gb300 import workload

from .test_oracle_pins import (_bf16_rne_by_bits, _rand_layer, _rand_x, _torch_dequant,
                               _torch_mx_quantize)


def _torch_roundtrip(v: np.ndarray) -> np.ndarray:
    """MXFP8 round trip of rows of values (exactly float32-representable)."""
    codes, scales = _torch_mx_quantize(v.astype(np.float32))
    return _torch_dequant(codes, scales).numpy()


def _bf16_round(v: np.ndarray) -> np.ndarray:
    bits = np.array([_bf16_rne_by_bits(float(a)) for a in v.ravel()], dtype=np.uint16)
    return workload.bf16_bits_to_f32(bits).astype(np.float64).reshape(v.shape)


def _torch_variant(layer, x_bits, ids, w, round_h, mx_acts):
    Wg = _torch_dequant(layer.gate_codes, layer.gate_scales)
    Wu = _torch_dequant(layer.up_codes, layer.up_scales)
    Wd = _torch_dequant(layer.down_codes, layer.down_scales)
    xs = workload.bf16_bits_to_f32(x_bits).astype(np.float64)
    y = np.zeros(xs.shape)
    for t in range(xs.shape[0]):
        xt = _torch_roundtrip(xs[t:t + 1])[0] if mx_acts else xs[t]
        xt = torch.from_numpy(xt)
        for j in range(ids.shape[1]):
            e = ids[t, j]
            hv = (torch.nn.functional.silu(Wg[e] @ xt) * (Wu[e] @ xt)).numpy()
            if round_h:
                hv = _bf16_round(hv)
            if mx_acts:
                hv = _torch_roundtrip(hv[None])[0]
            y[t] += float(w[t, j]) * (Wd[e] @ torch.from_numpy(hv)).numpy()
    return y


@pytest.mark.parametrize("round_h,mx_acts", [(1, 0), (0, 0), (1, 1)])
def test_variant_matches_torch(round_h, mx_acts):
    H, I, E, k = 64, 96, 3, 2
    layer = _rand_layer(H, I, E, 90)
    x = _rand_x(3, H, 91)
    ids = np.array([[0, 2], [1, 0], [2, 1]], dtype=np.int32)
    w = np.array([[0.6, 0.4], [0.3, 0.7], [0.5, 0.5]], dtype=np.float32)
    y = oracle.moe_layer_variant(layer, x, ids, w, bool(round_h), bool(mx_acts))
    np.testing.assert_allclose(y, _torch_variant(layer, x, ids, w, round_h, mx_acts),
                               rtol=1e-12, atol=1e-12)
    if round_h and not mx_acts:  # the layer itself
        np.testing.assert_array_equal(y, oracle.moe_layer(layer, x, ids, w)[0])


def _compact_layer(shape, ids, seed=0):
    """Oracle layer holding only the experts `ids` uses, ids renumbered to it."""
    used = np.unique(ids)
    g, u, d = workload.all_weights(shape, seed=seed, experts=used)
    layer = oracle.QuantizedLayer.from_fp32(g, u, d)
    return layer, np.searchsorted(used, ids).astype(np.int32), (g, u, d)


def study(B=8, batch=321):
    """Relative L2 errors of the two paths against both references (Q30 shapes)."""
    s = workload.SHAPES["q30"]
    x, ids, w = workload.tokens(s, B, batch=batch)
    layer, cids, (g, u, d) = _compact_layer(s, ids)
    wd = oracle.moe_layer_variant(layer, x, cids, w, True, False)
    cl = oracle.moe_layer_variant(layer, x, cids, w, True, True)
    ref_mx = oracle.moe_layer_variant(layer, x, cids, w, False, False)
    xs = torch.from_numpy(workload.bf16_bits_to_f32(x).astype(np.float64))
    ref_fp = torch.zeros((B, s.H), dtype=torch.float64)
    G, U, D = (torch.from_numpy(a).to(torch.float64) for a in (g, u, d))
    for t in range(B):
        for j in range(s.top_k):
            e = cids[t, j]
            hv = torch.nn.functional.silu(G[e] @ xs[t]) * (U[e] @ xs[t])
            ref_fp[t] += float(w[t, j]) * (D[e] @ hv)
    ref_fp = ref_fp.numpy()
    err = lambda a, r: float(np.linalg.norm(a - r) / np.linalg.norm(r))
    out = {}
    for name, ref in (("same MXFP8 weights", ref_mx), ("FP32 weights", ref_fp)):
        out[name] = {"warp_decode": err(wd, ref), "round_trip": err(cl, ref),
                     "ratio": err(cl, ref) / err(wd, ref),
                     "bf16_outputs_ratio": err(_bf16_round(cl), ref) / err(_bf16_round(wd), ref)}
    return out


# token batches of the study: (tokens, batch index of the seeded generator)
STUDY_BATCHES = ((8, 321), (4, 322), (4, 323), (4, 324))
PAGES_RATIO = 1.4  # [§Improved accuracy]: 1.4x closer to the FP32 reference


def test_warp_decode_is_closer_than_the_activation_round_trip():
    """Four independent token batches (20 tokens, about 110 experts): on every
    batch warp decode is closer to both references than the activation round
    trip, and against the unquantised FP32 weights the mean factor lies within
    15 % of the pages' 1.4; the per-batch spread is printed."""
    ratios = []
    for B, batch in STUDY_BATCHES:
        res = study(B, batch)
        print(B, batch, {k: round(v["ratio"], 3) for k, v in res.items()})
        # the direction the pages report, under both readings of the reference
        assert res["same MXFP8 weights"]["ratio"] > 1.0
        assert res["FP32 weights"]["ratio"] > 1.0
        ratios.append(res["FP32 weights"]["ratio"])
    mean = float(np.mean(ratios))
    print("FP32-weights ratio per batch", [round(r, 3) for r in ratios], "mean", round(mean, 3))
    assert abs(mean - PAGES_RATIO) <= 0.15 * PAGES_RATIO
