"""GPU router (moe_route) and the layer from router logits (moe_layer_routed).

The experts are chosen on the FP32 logits themselves on both sides (the oracle
in FP64 from the same FP32 values), so the chosen ids must match exactly; the
weights differ only by FP32 rounding of the exponentials (rtol 1e-6).
"""
import numpy as np
import pytest
import torch

import oracle
from output_centric_expert_gb300 import ops, workload

from ._layers import Layer, parity_stats
from .test_parity_gpu import MAX_ABS, MIN_COS, _dev

pytestmark = pytest.mark.gpu


def _route_gpu(shape, logits):
    B = logits.shape[0]
    ids = torch.empty((B, shape.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((B, shape.top_k), dtype=torch.float32, device="cuda")
    ops.moe_route(ops.make_shape(shape.H, shape.I, shape.E, shape.top_k), _dev(logits), ids, w)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("name,B,routing", [("q30", 64, "uniform"), ("q30", 64, "skewed"),
                                            ("dsv3", 33, "uniform"), ("tiny", 5, "uniform")])
def test_route_matches_oracle(name, B, routing):
    s = workload.SHAPES[name]
    L = workload.logits(s, B, batch=40, routing=routing)
    ids, w = _route_gpu(s, L)
    rids, rw = oracle.route(L, s.top_k)
    assert np.array_equal(ids, rids)
    np.testing.assert_allclose(w, rw, rtol=1e-6)


def test_route_ties_and_k_equals_e():
    s = workload.LayerShape(256, 128, 40, 32)  # top_k = 32 = a full warp of choices
    rng = np.random.default_rng(3)
    L = (np.round(rng.standard_normal((9, 40)) * 2) / 2).astype(np.float32)  # many equal logits
    L[0] = 0.0  # all equal
    ids, w = _route_gpu(s, L)
    rids, rw = oracle.route(L, s.top_k)
    assert np.array_equal(ids, rids)
    np.testing.assert_allclose(w, rw, rtol=1e-6)
    s2 = workload.LayerShape(256, 128, 8, 8)  # k = E
    L2 = rng.standard_normal((3, 8)).astype(np.float32)
    ids2, w2 = _route_gpu(s2, L2)
    rids2, rw2 = oracle.route(L2, 8)
    assert np.array_equal(ids2, rids2)
    np.testing.assert_allclose(w2, rw2, rtol=1e-6)


@pytest.fixture(scope="module")
def q30():
    return Layer(workload.SHAPES["q30"])


# B=1, 2, 4 and 32 run moe_down with 1 x 8, 2 x 4, 4 x 2 and 8 x 1 outputs x units per lane;
# with ids_out/wts_out given the routing is computed once into them (the gate/up kernel then
# runs as a programmatic dependent of the router; from 26 tokens the grouped one, from 40 the
# grouped down too), without them every CTA of both kernels routes its token itself
@pytest.mark.parametrize("B", [1, 2, 4, 26, 32, 64])
@pytest.mark.parametrize("keep_routing", [True, False])
def test_layer_from_logits(q30, B, keep_routing):
    """moe_layer_routed == moe_layer fed moe_route's routing (bit for bit) when
    it keeps the routing; without ids_out it equals the per-token kernels fed
    that routing bit for bit (moe_layer itself switches to the expert-grouped
    kernels at larger batches, which agree to FP32 rounding order); and it
    matches the oracle layer fed the oracle's routing."""
    s = q30.shape
    x, _, _ = workload.tokens(s, B, batch=60 + B)
    L = workload.logits(s, B, batch=60 + B)
    xd, Ld = _dev(x.view(np.int16)), _dev(L)
    h = torch.empty((B, s.top_k, s.I), dtype=torch.int16, device="cuda")
    y = torch.empty((B, s.H), dtype=torch.float32, device="cuda")
    ids_out = torch.empty((B, s.top_k), dtype=torch.int32, device="cuda")
    w_out = torch.empty((B, s.top_k), dtype=torch.float32, device="cuda")
    if keep_routing:
        ops.moe_layer_routed(q30.dev, xd, Ld, h, y, ids_out, w_out)
    else:
        ops.moe_layer_routed(q30.dev, xd, Ld, h, y)
    ids, w = _route_gpu(s, L)
    y2 = torch.empty_like(y)
    h2 = torch.empty_like(h)
    if keep_routing:
        ops.moe_layer(q30.dev, xd, _dev(ids), _dev(w), h2, y2)
    else:
        ops.moe_gate_up(q30.dev, xd, _dev(ids), h2)
        ops.moe_down(q30.dev, h2, _dev(ids), _dev(w), y2)
    torch.cuda.synchronize()
    if keep_routing:
        assert np.array_equal(ids_out.cpu().numpy(), ids)
        assert np.array_equal(w_out.cpu().numpy(), w)
    assert np.array_equal(y.cpu().numpy(), y2.cpu().numpy())
    assert np.array_equal(h.cpu().numpy(), h2.cpu().numpy())
    rids, rw = oracle.route(L, s.top_k)
    y_ref, _ = oracle.moe_layer(q30.ref, x, rids, rw.astype(np.float32))
    d, cos = parity_stats(y.cpu().numpy(), y_ref)
    assert d <= MAX_ABS and cos >= MIN_COS, (d, cos)
