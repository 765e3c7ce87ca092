"""GPU parity of the expert-grouped moe_gate_up (moe_gate_up_grouped) against the oracle.

The grouped kernel gives every (expert, 8 neurons) warp all the (token, slot)
pairs routed to that expert as tensor-core MMA columns, 8 per pass. The
cases below cover one and several passes over the weights (a hot expert),
whole items and half-items split over H, several items per CTA, duplicate
ids, invalid ids, the shapes of the target layers and the shapes the kernel
refuses.
"""
import numpy as np
import pytest
import torch

import oracle
from output_centric_expert_gb300 import ops, workload
from tests._layers import Layer
from tests.test_parity_gpu import _check_h, _dev

pytestmark = pytest.mark.gpu

_SENTINEL = 0x7FC1  # a BF16 NaN no kernel writes: shows outputs left unwritten


def _grouped(layer, x, ids):
    B = x.shape[0]
    h = torch.full((B, layer.shape.top_k, layer.shape.I), _SENTINEL, dtype=torch.int16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.moe_gate_up_grouped(layer.dev, _dev(x.view(np.int16)), _dev(ids), h, err)
    torch.cuda.synchronize()
    return h.cpu().numpy().view(np.uint16), int(err.item())


def _h_ref(layer, x, ids):
    _, h_ref, bad = oracle.moe_layer(layer.ref, x, ids, np.ones(ids.shape, np.float32), return_h=True)
    return h_ref, bad


@pytest.fixture(scope="module")
def q30():
    return Layer(workload.SHAPES["q30"])


@pytest.fixture(scope="module")
def tiny():
    return Layer(workload.SHAPES["tiny"])


@pytest.mark.parametrize("B,routing", [(1, "uniform"), (8, "uniform"), (32, "uniform"), (64, "skewed"),
                                       (96, "uniform")])
def test_grouped_q30_every_token(q30, B, routing):
    """Qwen-3-30B-A3B-shaped layer: every intermediate of every token. Skewed
    routing at B=64 puts more than 16 pairs on the hot experts (several passes);
    96 tokens put 6 pairs on an expert on average."""
    x, ids, _ = workload.tokens(q30.shape, B, routing=routing, batch=B)
    h, err = _grouped(q30, x, ids)
    h_ref, _ = _h_ref(q30, x, ids)
    assert err == 0
    _check_h(h, h_ref)


def test_grouped_hot_expert_with_duplicates_several_passes(tiny):
    """Every slot of 40 tokens on expert 3 (duplicate ids in each token): 80 pairs
    on one expert, 10 passes of 8 columns over its rows; the other experts idle."""
    B = 40
    x, _, _ = workload.tokens(tiny.shape, B, batch=21)
    ids = np.full((B, 2), 3, dtype=np.int32)
    h, err = _grouped(tiny, x, ids)
    h_ref, _ = _h_ref(tiny, x, ids)
    assert err == 0
    assert np.array_equal(h[:, 0], h[:, 1])  # a duplicate slot is the same pair twice
    _check_h(h, h_ref)


def test_grouped_several_items_per_cta(tiny):
    """1600 tokens of the tiny layer: 3200 pairs in 8-column passes make about
    800 work items, more than the persistent grid's CTAs, so CTAs run several
    whole items one after the other (rows of 256: one 8-block group, no
    half-items). Every intermediate against the oracle."""
    B = 1600
    x, ids, _ = workload.tokens(tiny.shape, B, batch=23)
    h, err = _grouped(tiny, x, ids)
    h_ref, _ = _h_ref(tiny, x, ids)
    assert err == 0
    _check_h(h, h_ref)


def test_grouped_invalid_ids(tiny):
    B = 24
    x, ids, _ = workload.tokens(tiny.shape, B, batch=7)
    ids = ids.copy()
    ids[3, 0] = 8      # == E
    ids[17, 1] = -1
    h, err = _grouped(tiny, x, ids)
    h_ref, bad = _h_ref(tiny, x, ids)
    assert bad == 2 and err == 1
    assert np.all(h[3, 0] == 0) and np.all(h[17, 1] == 0)
    _check_h(h, h_ref)


@pytest.mark.parametrize("B", [32, 29, 96, 128])
def test_grouped_result_of_a_token_does_not_depend_on_the_batch(q30, B):
    """Each (token, slot) column is an independent MMA column and every item
    sums the lower and the upper half of H separately, whether it runs whole,
    as a half-item split over two warps, so a token's intermediate is
    bit-identical alone (every half-item split) and in a batch (29 and 32
    tokens run half-item shares, 96 and 128 whole items)."""
    x, ids, _ = workload.tokens(q30.shape, B, batch=500 + B)
    h, _ = _grouped(q30, x, ids)
    for t in (0, 13, B // 2, B - 1):
        h1, _ = _grouped(q30, x[t:t + 1], ids[t:t + 1])
        assert np.array_equal(h1[0], h[t]), t


@pytest.mark.parametrize("name,E,B", [("q235", 8, 16), ("dsv3", 16, 4), ("mixtral", 8, 3)])
def test_grouped_shape_variants(name, E, B):
    """Qwen-3-235B-A22B-, DeepSeek-V3- and Mixtral-shaped rows with fewer experts:
    H=4096 and H=7168 stage 8 columns per pass (16 at H=2048), so 16 tokens on 8
    experts need several passes."""
    full = workload.SHAPES[name]
    s = workload.LayerShape(full.H, full.I, E, full.top_k)
    x, ids, _ = workload.tokens(s, B, batch=12)
    sample = sorted({0, B // 2, B - 1})
    layer = Layer(s, oracle_experts=np.unique(ids[sample]))
    h, err = _grouped(layer, x, ids)
    h_ref, _ = _h_ref(layer, x[sample], ids[sample])
    assert err == 0
    _check_h(h[sample], h_ref)
    assert not np.any(h == _SENTINEL)


@pytest.mark.parametrize("H,I,E,k,B", [
    (256, 128, 8, 8, 4),   # top_k = E
    (512, 64, 3, 3, 2),    # one CTA of neurons per expert, top_k = E
    (768, 192, 5, 3, 9),   # three neuron tiles, odd batch
])
def test_grouped_small_shapes(H, I, E, k, B):
    layer = Layer(workload.LayerShape(H, I, E, k), seed=H + I)
    x, ids, _ = workload.tokens(layer.shape, B, seed=7)
    h, _ = _grouped(layer, x, ids)
    h_ref, _ = _h_ref(layer, x, ids)
    _check_h(h, h_ref)


@pytest.mark.parametrize("H,I,E", [(96, 160, 2), (2080, 800, 2), (2048, 96, 2), (256, 64, 257)])
def test_grouped_refuses_unsupported_shapes(H, I, E):
    layer = Layer(workload.LayerShape(H, I, E, 1), seed=1)
    x, ids, _ = workload.tokens(layer.shape, 1, seed=3)
    with pytest.raises(ops.WarpDecodeError) as exc:
        _grouped(layer, x, ids)
    assert exc.value.status == 5  # MOE_ERR_UNSUPPORTED
