"""GPU parity of the expert-grouped moe_down (moe_down_grouped) against the oracle.

The grouped kernel gives each CTA 16 output rows for every token of the batch;
its warps take the batch's routed experts in turn, stream each expert's 16
down rows once and multiply them on the tensor cores against up to 8 routed
pairs per pass. The cases below cover one and several passes over an
expert's rows (a hot expert), duplicate ids within a token (two MMA columns of
one token), invalid ids, tokens with nothing routed, a NaN scale, the row
shapes of the target layers, every batch size the layer hands it, and the
shapes and batches it refuses.
"""
import numpy as np
import pytest
import torch

import oracle
from output_centric_expert_gb300 import ops, workload
from tests._layers import Layer, parity_stats
from tests.test_parity_gpu import MAX_ABS, MIN_COS, _check_y, _dev

pytestmark = pytest.mark.gpu

# moe_down fed the oracle's own intermediate: only the FP32 summation order
# differs from the oracle (y ~ 2 at unit scale, sums of top_k * I terms)
DOWN_ABS = 1e-4


def _down(layer, h_bits, ids, w, grouped=True, err=None):
    B = ids.shape[0]
    y = torch.full((B, layer.shape.H), float("nan"), dtype=torch.float32, device="cuda")
    fn = ops.moe_down_grouped if grouped else ops.moe_down
    fn(layer.dev, _dev(h_bits.view(np.int16)), _dev(ids), _dev(w), y, err)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def _gpu_h(layer, x, ids):
    B = x.shape[0]
    h = torch.empty((B, layer.shape.top_k, layer.shape.I), dtype=torch.int16, device="cuda")
    ops.moe_gate_up(layer.dev, _dev(x.view(np.int16)), _dev(ids), h)
    torch.cuda.synchronize()
    return h.cpu().numpy().view(np.uint16)


@pytest.fixture(scope="module")
def q30():
    return Layer(workload.SHAPES["q30"])


@pytest.fixture(scope="module")
def small():
    """A small layer the grouped kernel takes (I % 256 == 0): H=64, I=256, E=6, top-3."""
    return Layer(workload.LayerShape(64, 256, 6, 3), seed=5)


@pytest.mark.parametrize("B,routing", [(1, "uniform"), (16, "uniform"), (32, "uniform"),
                                       (32, "skewed"), (64, "skewed")])
def test_grouped_down_on_oracle_intermediate_every_token(q30, B, routing):
    """Qwen-3-30B-A3B-shaped layer fed the oracle's own BF16 intermediate: every
    output of every token within FP32 summation error of the oracle. Skewed
    routing puts more than 8 pairs on the hot experts (several passes)."""
    x, ids, w = workload.tokens(q30.shape, B, routing=routing, batch=300 + B)
    y_ref, h_ref, _ = oracle.moe_layer(q30.ref, x, ids, w, return_h=True)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = _down(q30, h_ref, ids, w, err=err)
    d, cos = parity_stats(y, y_ref)
    assert d <= DOWN_ABS and cos >= MIN_COS, (d, cos)
    assert int(err.item()) == 0


def test_grouped_down_matches_per_token_down_every_batch(q30):
    """Same intermediate into both down kernels at every batch the layer sweep
    uses (and 96 tokens, near the batch this shape's shared memory allows):
    they differ in FP32 rounding order only."""
    for B, routing in [(b, r) for r in ("uniform", "skewed") for b in (1, 2, 4, 8, 16, 32, 64)] + \
            [(96, "uniform")]:
        x, ids, w = workload.tokens(q30.shape, B, routing=routing, batch=400 + B)
        h = _gpu_h(q30, x, ids)
        yg = _down(q30, h, ids, w)
        yp = _down(q30, h, ids, w, grouped=False)
        assert np.all(np.isfinite(yg)), (B, routing)
        d, cos = parity_stats(yg, yp.astype(np.float64))
        assert d <= DOWN_ABS and cos >= MIN_COS, (B, routing, d, cos)


@pytest.mark.parametrize("B", [48, 96])
def test_grouped_down_layer_sampled_tokens(q30, B):
    """The whole layer at batches where it runs the grouped down kernel (after
    the grouped gate/up kernel at both), against the oracle on sampled tokens."""
    x, ids, w = workload.tokens(q30.shape, B, batch=500 + B)
    assert ops.layer_down_kernel(q30.sh, B, q30.dev) == "grouped"
    h = torch.empty((B, 8, q30.shape.I), dtype=torch.int16, device="cuda")
    y = torch.empty((B, q30.shape.H), dtype=torch.float32, device="cuda")
    ops.moe_layer(q30.dev, _dev(x.view(np.int16)), _dev(ids), _dev(w), h, y)
    torch.cuda.synchronize()
    sample = sorted({0, 1, B // 3, B // 2, B - 2, B - 1})
    y_ref, _ = oracle.moe_layer(q30.ref, x[sample], ids[sample], w[sample])
    _check_y(y.cpu().numpy()[sample], y_ref)


def test_layer_switches_down_kernel_at_2_5e_pairs(q30):
    """moe_layer's y equals moe_down's below 2 * B * top_k = 5E and
    moe_down_grouped's from there on (Qwen-3-30B-A3B shape: 40 tokens), bit for
    bit, on the intermediate the layer itself produced."""
    for B in (39, 40):
        x, ids, w = workload.tokens(q30.shape, B, batch=600 + B)
        h = torch.empty((B, 8, q30.shape.I), dtype=torch.int16, device="cuda")
        y = torch.empty((B, q30.shape.H), dtype=torch.float32, device="cuda")
        ops.moe_layer(q30.dev, _dev(x.view(np.int16)), _dev(ids), _dev(w), h, y)
        torch.cuda.synchronize()
        hb = h.cpu().numpy().view(np.uint16)
        want = _down(q30, hb, ids, w, grouped=(2 * B * 8 >= 5 * 128))
        assert ops.layer_down_kernel(q30.sh, B, q30.dev) == ("grouped" if 2 * B * 8 >= 5 * 128 else "per_token")
        assert np.array_equal(y.cpu().numpy(), want), B


def test_layer_switches_down_kernel_for_long_intermediate_rows():
    """Mixtral-shaped layer (I = 14336, three and a half times H): moe_layer's y
    equals moe_down's at 4 tokens (8 pairs on 8 experts) and moe_down_grouped's
    from 4 * B * top_k >= 5E (5 tokens), bit for bit, on the intermediate the
    layer itself produced; the gate/up step stays per-token below 2 * B * top_k
    = 3E (6 tokens)."""
    s = workload.SHAPES["mixtral"]
    layer = Layer(s, oracle_experts=[])
    for B, want in ((4, ("per_token", "per_token")), (5, ("per_token", "grouped")),
                    (6, ("grouped", "grouped"))):
        assert (ops.layer_gate_up_kernel(layer.sh, B), ops.layer_down_kernel(layer.sh, B)) == want
        x, ids, w = workload.tokens(s, B, batch=650 + B)
        h = torch.empty((B, s.top_k, s.I), dtype=torch.int16, device="cuda")
        y = torch.empty((B, s.H), dtype=torch.float32, device="cuda")
        ops.moe_layer(layer.dev, _dev(x.view(np.int16)), _dev(ids), _dev(w), h, y)
        torch.cuda.synchronize()
        yd = _down(layer, h.cpu().numpy().view(np.uint16), ids, w, grouped=(want[1] == "grouped"))
        assert np.array_equal(y.cpu().numpy(), yd), B


@pytest.mark.parametrize("B,routing,batch", [(32, "skewed", 0), (32, "skewed", 3), (16, "skewed", 1),
                                             (32, "uniform", 0), (40, "uniform", 2)])
def test_host_entry_point_chooses_from_its_ids(q30, B, routing, batch):
    """moe_layer_host picks its kernels from the batch's own ids (pairs per used
    expert): a skewed batch of 32 tokens runs both grouped kernels although
    moe_layer, which decides on B, runs the per-token down kernel there. Its y equals,
    bit for bit, the kernels it reports run one after the other on the same
    device inputs, and the oracle on sampled tokens."""
    x, ids, w = workload.tokens(q30.shape, B, routing=routing, batch=batch)
    gu, dn = ops.layer_host_kernels(q30.sh, ids, q30.dev)
    if routing == "skewed" and B == 32:
        assert (gu, dn) == ("grouped", "grouped")
    if routing == "uniform":
        assert (gu, dn) == (ops.layer_gate_up_kernel(q30.sh, B), ops.layer_down_kernel(q30.sh, B))
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    xh, idh, wh = pin(x.view(np.int16)), pin(ids), pin(w)
    yh = torch.full((B, q30.shape.H), float("nan"), dtype=torch.float32).pin_memory()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    dev = dict(x_dev=torch.empty_like(xh, device="cuda"), ids_dev=torch.empty_like(idh, device="cuda"),
               wts_dev=torch.empty_like(wh, device="cuda"),
               h_dev=torch.empty((B, 8, q30.shape.I), dtype=torch.int16, device="cuda"),
               y_dev=torch.empty((B, q30.shape.H), dtype=torch.float32, device="cuda"))
    ops.moe_layer_host(q30.dev, xh, idh, wh, y_host=yh, err_flag=err, **dev)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    h = torch.empty((B, 8, q30.shape.I), dtype=torch.int16, device="cuda")
    (ops.moe_gate_up_grouped if gu == "grouped" else ops.moe_gate_up)(
        q30.dev, _dev(x.view(np.int16)), _dev(ids), h)
    torch.cuda.synchronize()
    want = _down(q30, h.cpu().numpy().view(np.uint16), ids, w, grouped=(dn == "grouped"))
    assert np.array_equal(yh.numpy(), want)
    sample = sorted({0, B // 2, B - 1})
    y_ref, _ = oracle.moe_layer(q30.ref, x[sample], ids[sample], w[sample])
    _check_y(yh.numpy()[sample], y_ref)


def test_grouped_down_deterministic(q30):
    x, ids, w = workload.tokens(q30.shape, 48, routing="skewed", batch=7)
    h = _gpu_h(q30, x, ids)
    y1 = _down(q30, h, ids, w)
    y2 = _down(q30, h, ids, w)
    assert np.array_equal(y1, y2)


def test_hot_expert_duplicates_invalid_ids_and_empty_tokens(small):
    """40 tokens: slot 0 of every token on expert 2 (40 pairs: 5 passes of 8
    columns), token 3 routed to expert 4 in all three slots and token 9 twice
    to expert 2 (duplicate ids: columns of one token in neighbouring lanes),
    token 5 with only invalid ids (its outputs are 0), two more invalid ids,
    and a zero routing weight."""
    s = small.shape
    B = 40
    x, ids, w = workload.tokens(s, B, batch=21)
    ids = ids.copy()
    w = w.copy()
    ids[:, 0] = 2
    ids[3, :] = 4
    ids[9, 1] = 2
    ids[5, :] = [-1, 6, 99]
    ids[17, 2] = -7
    ids[30, 1] = 6
    w[11, 1] = 0.0
    y_ref, h_ref, bad = oracle.moe_layer(small.ref, x, ids, w, return_h=True)
    assert bad == 5
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = _down(small, h_ref, ids, w, err=err)
    assert int(err.item()) == 1
    assert np.all(y[5] == 0.0)
    d, cos = parity_stats(y, y_ref)
    assert d <= DOWN_ABS, d
    # and the layer as a whole (2 * B * top_k >= 5E: grouped down)
    h = torch.empty((B, s.top_k, s.I), dtype=torch.int16, device="cuda")
    yl = torch.empty((B, s.H), dtype=torch.float32, device="cuda")
    err.zero_()
    ops.moe_layer(small.dev, _dev(x.view(np.int16)), _dev(ids), _dev(w), h, yl, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 1
    keep = [t for t in range(B) if t != 5]
    _check_y(yl.cpu().numpy()[keep], y_ref[keep])


def test_all_tokens_on_one_expert_every_slot(small):
    """Every slot of 128 tokens on expert 1: 384 pairs, 48 passes over one
    expert's rows; every other expert idle."""
    s = small.shape
    B = 128
    x, _, _ = workload.tokens(s, B, batch=22)
    ids = np.full((B, s.top_k), 1, dtype=np.int32)
    w = np.tile(np.array([[0.5, 0.3, 0.2]], np.float32), (B, 1))
    y_ref, h_ref, _ = oracle.moe_layer(small.ref, x, ids, w, return_h=True)
    y = _down(small, h_ref, ids, w)
    d, _ = parity_stats(y, y_ref)
    assert d <= DOWN_ABS, d


def test_nan_scale_propagates_to_its_outputs(small):
    s = small.shape
    B = 4
    x, ids, w = workload.tokens(s, B, batch=23)
    ids = ids.copy()
    ids[0] = [3, 0, 1]
    ids[1:, :] = np.where(ids[1:] == 3, 5, ids[1:])  # only token 0 uses expert 3
    _, h_ref, _ = oracle.moe_layer(small.ref, x, ids, w, return_h=True)
    y_ok = _down(small, h_ref, ids, w)
    d_scales = small.dev.tensors[3].view(s.E, s.H, s.I // 32)
    saved = int(d_scales[3, 7, 2].item())
    d_scales[3, 7, 2] = 0xFF
    try:
        y = _down(small, h_ref, ids, w)
    finally:
        d_scales[3, 7, 2] = saved
    assert np.isnan(y[0, 7])
    assert np.array_equal(np.delete(y[0], 7), np.delete(y_ok[0], 7))
    assert np.array_equal(y[1:], y_ok[1:])


@pytest.mark.parametrize("name,E,B", [("q235", 16, 24), ("dsv3", 16, 16), ("mixtral", 4, 12)])
def test_grouped_down_target_row_shapes(name, E, B):
    """Rows of 1536 (6 steps), 2048 (8 steps) and 14336 (56 steps) elements,
    with H = 4096 and 7168 (256 and 448 CTAs), fewer experts than the models."""
    full = workload.SHAPES[name]
    s = workload.LayerShape(full.H, full.I, E, full.top_k)
    x, ids, w = workload.tokens(s, B, batch=31)
    sample = sorted({0, B // 2, B - 1})
    layer = Layer(s, oracle_experts=np.unique(ids))
    h = _gpu_h(layer, x, ids)
    yg = _down(layer, h, ids, w)
    yp = _down(layer, h, ids, w, grouped=False)
    d, cos = parity_stats(yg, yp.astype(np.float64))
    assert d <= 4 * DOWN_ABS and cos >= MIN_COS, (d, cos)
    y_ref, _ = oracle.moe_layer(layer.ref, x[sample], ids[sample], w[sample])
    _check_y(yg[sample], y_ref)


def test_grouped_down_refuses_what_it_cannot_take(q30):
    """I % 256 != 0, E > 256, B > 128: MOE_ERR_UNSUPPORTED and nothing written;
    the layer then keeps the per-token kernel."""
    s = workload.LayerShape(64, 160, 4, 2)
    layer = Layer(s, seed=9)
    x, ids, w = workload.tokens(s, 8, batch=1)
    y = torch.full((8, s.H), 3.0, dtype=torch.float32, device="cuda")
    h = torch.zeros((8, 2, s.I), dtype=torch.int16, device="cuda")
    with pytest.raises(ops.WarpDecodeError) as ei:
        ops.moe_down_grouped(layer.dev, h, _dev(ids), _dev(w), y)
    assert ei.value.status == 5
    torch.cuda.synchronize()
    assert bool(torch.all(y == 3.0))
    assert ops.layer_down_kernel(layer.sh, 8, layer.dev) == "per_token"
    assert ops.layer_down_kernel(q30.sh, 129) == "per_token"
    assert ops.layer_down_kernel(ops.make_shape(2048, 768, 257, 8), 64) == "per_token"
    B = 129
    ids = torch.zeros((B, 8), dtype=torch.int32, device="cuda")
    with pytest.raises(ops.WarpDecodeError) as ei:
        ops.moe_down_grouped(q30.dev, torch.zeros((B, 8, 768), dtype=torch.int16, device="cuda"),
                             ids, torch.zeros((B, 8), dtype=torch.float32, device="cuda"),
                             torch.zeros((B, 2048), dtype=torch.float32, device="cuda"))
    assert ei.value.status == 5


@pytest.mark.parametrize("world,B", [(2, 32), (3, 64), (32, 8)])
def test_expert_parallel_shards_sum_to_the_layer(q30, world, B):
    """The layer split over `world` expert shards on one device, one shard at a
    time (moe_local_ids, then moe_layer on the shard's experts with no error
    flag), summed on the host: within the parity bar of the whole layer and of
    the oracle. 32 shards hold 4 experts each, fewer than top_k."""
    from output_centric_expert_gb300 import expert_parallel as ep
    s = q30.shape
    x, ids, w = workload.tokens(s, B, batch=900 + B)
    xd, idd, wd = _dev(x.view(np.int16)), _dev(ids), _dev(w)
    total = torch.zeros((B, s.H), dtype=torch.float64, device="cuda")
    local = torch.empty_like(idd)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    covered = 0
    for r in range(world):
        first, count = ep.shard_range(s.E, r, world)
        part = ep.shard_packed(q30.packed, s, first, count)
        shard = ops.DeviceWeights(ops.make_shape(s.H, s.I, count, s.top_k), part)
        h = torch.empty((B, s.top_k, s.I), dtype=torch.int16, device="cuda")
        y = torch.empty((B, s.H), dtype=torch.float32, device="cuda")
        ep.ep_layer(shard, xd, idd, wd, h, y, first, count, global_E=s.E, local_ids=local,
                    err_flag=err, all_reduce=False)
        torch.cuda.synchronize()
        lid = local.cpu().numpy()
        want = np.where((ids >= first) & (ids < first + count), ids - first, -1)
        assert np.array_equal(lid, want)
        covered += int((lid >= 0).sum())
        total += y.double()
    assert covered == B * s.top_k and int(err.item()) == 0
    h = torch.empty((B, s.top_k, s.I), dtype=torch.int16, device="cuda")
    y_all = torch.empty((B, s.H), dtype=torch.float32, device="cuda")
    ops.moe_layer(q30.dev, xd, idd, wd, h, y_all)
    torch.cuda.synchronize()
    # a shard has fewer experts, so the layer may choose the other gate/up
    # kernel for it than for the whole layer (an intermediate can then differ
    # by one BF16 step): the layer's parity bar applies
    d, cos = parity_stats(total.cpu().numpy(), y_all.cpu().numpy().astype(np.float64))
    assert d <= MAX_ABS and cos >= MIN_COS, (d, cos)
    sample = [0, B - 1]
    y_ref, _ = oracle.moe_layer(q30.ref, x[sample], ids[sample], w[sample])
    _check_y(total.cpu().numpy()[sample], y_ref)


def test_local_ids_flag_ids_outside_the_global_range(q30):
    ids = torch.tensor([[0, 5, 127, 128], [-1, 64, 63, 3]], dtype=torch.int32, device="cuda")
    local = torch.empty_like(ids)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    sh = ops.make_shape(2048, 768, 128, 4)
    ops.moe_local_ids(sh, ids, 64, 64, local, err)
    torch.cuda.synchronize()
    assert local.cpu().tolist() == [[-1, -1, 63, -1], [-1, 0, -1, -1]]
    assert int(err.item()) == 1
    with pytest.raises(ops.WarpDecodeError):
        ops.moe_local_ids(sh, ids, 64, 65, local)
