"""GPU parity: the CUDA path (through the C ABI) against the FP64 CPU oracle.

Bar: per token, max |y_gpu - y_oracle| <= 4e-3 and cosine >= 0.99999 for
unit-scale inputs (x ~ N(0,1), W ~ N(0, 0.05^2)). The BF16 intermediate h is
also compared. The kernel rounds silu(g)*u from FP32-accumulated g and u (the
pages keep accumulators in FP32), the oracle from exact ones, so a code may
differ by one BF16 step where the two values straddle a rounding boundary, and
by the FP32 accumulation error where the dot product cancels: at most about
30 * 2^-24 * sum|x*w| ~ 1e-4 absolute for H <= 4096 at unit scale. Codes must
agree in all but a small fraction of places.
"""
import numpy as np
import pytest
import torch

import oracle
from output_centric_expert_gb300 import ops, workload

from ._layers import Layer, parity_stats

pytestmark = pytest.mark.gpu

MAX_ABS = 4e-3
MIN_COS = 0.99999


def _dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return t.view(dtype) if dtype is not None else t


def _run_layer(layer: Layer, x, ids, w, with_err=False):
    B = x.shape[0]
    k = layer.shape.top_k
    xd, idd, wd = _dev(x.view(np.int16)), _dev(ids), _dev(w)
    h = torch.empty((B, k, layer.shape.I), dtype=torch.int16, device="cuda")
    y = torch.empty((B, layer.shape.H), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.moe_layer(layer.dev, xd, idd, wd, h, y, err)
    torch.cuda.synchronize()
    out = (y.cpu().numpy(), h.cpu().numpy().view(np.uint16))
    return out + (int(err.item()),) if with_err else out


def _bf16_vals(bits):
    return workload.bf16_bits_to_f32(bits).astype(np.float64)


H_ABS = 2e-4  # FP32 accumulation error of g, u carried through silu(g)*u


def _check_h(h_gpu, h_ref, max_frac=0.01):
    diff = h_gpu != h_ref
    frac = float(diff.mean()) if diff.size else 0.0
    assert frac <= max_frac, f"{frac:.4%} of intermediate codes differ"
    if diff.any():
        vg, vr = _bf16_vals(h_gpu[diff]), _bf16_vals(h_ref[diff])
        allowed = 2.0**-7 * np.maximum(np.abs(vg), np.abs(vr)) + H_ABS
        worst = float(np.max(np.abs(vg - vr) - allowed))
        assert worst <= 0, f"an intermediate differs beyond one BF16 step + {H_ABS} (by {worst:.3e})"


def _check_y(y_gpu, y_ref):
    d, cos = parity_stats(y_gpu, y_ref)
    assert d <= MAX_ABS, f"max|dy| = {d:.3e}"
    assert cos >= MIN_COS, f"min cosine = {cos:.8f}"
    return d, cos


# ------------------------------------------------------------ fixtures ------

@pytest.fixture(scope="module")
def tiny():
    return Layer(workload.SHAPES["tiny"])


@pytest.fixture(scope="module")
def q30():
    return Layer(workload.SHAPES["q30"])


# ------------------------------------------------------- the named configs --

def test_tiny_config_full(tiny):
    """H=256, I=128, E=8, top-2, B=1, seed 0: every output and intermediate."""
    x, ids, w = workload.tokens(tiny.shape, 1)
    y, h = _run_layer(tiny, x, ids, w)
    y_ref, h_ref, bad = oracle.moe_layer(tiny.ref, x, ids, w, return_h=True)
    assert bad == 0
    _check_y(y, y_ref)
    _check_h(h, h_ref)


# B covers every moe_down configuration the launcher picks for this shape:
# 1 output x 8 units per lane (B=1), 2 x 4 (B=2), 4 x 2 (B=4, in
# test_activation_scale_extremes), 8 x 1 as one wave (B=7) and as several
# waves (B=32, 64).
@pytest.mark.parametrize("B,routing", [(1, "uniform"), (2, "uniform"), (32, "uniform"), (64, "skewed"),
                                       (7, "uniform")])
def test_q30_layer_all_tokens(q30, B, routing):
    """Qwen-3-30B-A3B-shaped layer (H=2048, I=768, E=128, top-8), every token."""
    x, ids, w = workload.tokens(q30.shape, B, routing=routing, batch=B)
    y, h = _run_layer(q30, x, ids, w)
    y_ref, h_ref, _ = oracle.moe_layer(q30.ref, x, ids, w, return_h=True)
    _check_y(y, y_ref)
    _check_h(h, h_ref)


def test_q30_down_kernel_alone_on_oracle_intermediate(q30):
    """moe_down fed the oracle's own BF16 intermediate: only summation order differs."""
    B = 16
    x, ids, w = workload.tokens(q30.shape, B, batch=99)
    y_ref, h_ref, _ = oracle.moe_layer(q30.ref, x, ids, w, return_h=True)
    y = torch.empty((B, q30.shape.H), dtype=torch.float32, device="cuda")
    ops.moe_down(q30.dev, _dev(h_ref.view(np.int16)), _dev(ids), _dev(w), y)
    torch.cuda.synchronize()
    d, _ = parity_stats(y.cpu().numpy(), y_ref)
    assert d <= 1e-4, d


def test_q30_gate_up_kernel_alone(q30):
    B = 8
    x, ids, _ = workload.tokens(q30.shape, B, batch=98)
    _, h_ref, _ = oracle.moe_layer(q30.ref, x, ids, np.ones(ids.shape, np.float32), return_h=True)
    h = torch.empty((B, q30.shape.top_k, q30.shape.I), dtype=torch.int16, device="cuda")
    ops.moe_gate_up(q30.dev, _dev(x.view(np.int16)), _dev(ids), h)
    torch.cuda.synchronize()
    _check_h(h.cpu().numpy().view(np.uint16), h_ref)


def _sample(B, n):
    """Up to n token indices spread over the batch, first and last included."""
    return sorted(set(np.linspace(0, B - 1, min(n, B)).round().astype(int).tolist()))


@pytest.mark.parametrize("B,routing", [(B, r) for r in ("uniform", "skewed") for B in (1, 2, 4, 8, 16, 32, 64)])
def test_sweep_config_sampled_tokens(q30, B, routing):
    """Every point of the Qwen-3-30B-A3B-shaped batch sweep, on the bench's first
    batch of that config: up to 8 tokens against the oracle."""
    x, ids, w = workload.tokens(q30.shape, B, routing=routing)
    y, h = _run_layer(q30, x, ids, w)
    sample = _sample(B, 8)
    y_ref, h_ref, _ = oracle.moe_layer(q30.ref, x[sample], ids[sample], w[sample], return_h=True)
    _check_y(y[sample], y_ref)
    _check_h(h[sample], h_ref)


Q235_BATCHES = (1, 16, 64)


@pytest.fixture(scope="module")
def q235():
    s = workload.SHAPES["q235"]
    need = set()
    for B in Q235_BATCHES:
        _, ids, _ = workload.tokens(s, B)
        need |= set(ids[_sample(B, 3)].ravel().tolist())
    return Layer(s, oracle_experts=sorted(need))


@pytest.mark.parametrize("B", Q235_BATCHES)
def test_q235_sampled_tokens(q235, B):
    """Qwen-3-235B-A22B-shaped layer (full size, all 128 experts on the device) at
    the configured batches; the oracle checks 3 tokens of each."""
    x, ids, w = workload.tokens(q235.shape, B)
    sample = _sample(B, 3)
    y, _ = _run_layer(q235, x, ids, w)
    y_ref, _ = oracle.moe_layer(q235.ref, x[sample], ids[sample], w[sample])
    _check_y(y[sample], y_ref)
    assert np.all(np.isfinite(y))


@pytest.mark.parametrize("name,E,B", [("dsv3", 16, 12), ("mixtral", 8, 6), ("mixtral", 8, 4),
                                      ("dsv3", 16, 1), ("mixtral", 8, 1), ("q235", 8, 1)])
def test_shape_variants(name, E, B):
    """DeepSeek-V3-shaped (H=7168: partial row segments) and Mixtral-shaped
    (I=14336: a 57 KB intermediate per token) layers, with fewer experts than the
    models have (parity depends on the row shapes, not on E). At B=1 moe_down
    runs 4 outputs x 2 units (H=7168) or 2 outputs x 4 units (H=4096) per lane."""
    full = workload.SHAPES[name]
    s = workload.LayerShape(full.H, full.I, E, full.top_k)
    x, ids, w = workload.tokens(s, B, batch=11)
    sample = sorted({0, B // 2, B - 1})
    layer = Layer(s, oracle_experts=np.unique(ids[sample]))
    y, h = _run_layer(layer, x, ids, w)
    y_ref, h_ref, _ = oracle.moe_layer(layer.ref, x[sample], ids[sample], w[sample], return_h=True)
    _check_y(y[sample], y_ref)
    _check_h(h[sample], h_ref)
    assert np.all(np.isfinite(y))


# ------------------------------------------------------------ edge cases ----

def _rand_layer_shape(H, I, E, k, seed=0):
    return Layer(workload.LayerShape(H, I, E, k), seed=seed)


@pytest.mark.parametrize("H,I,E,k,B", [
    (32, 32, 2, 1, 1),        # smallest shape: one scale block per row
    (2080, 800, 4, 2, 3),     # several load rounds with a ragged tail on both kernels
    (96, 160, 5, 3, 5),       # rows shorter than a warp's chunk span
    (544, 64, 3, 3, 2),       # top_k = E
    (256, 128, 8, 8, 4),      # tiny layer with k = E
    (96, 160, 5, 3, 128),     # H % 64 != 0 where 8 outputs per warp would leave outputs unwritten
    (96, 160, 5, 3, 10),      # 2 slots per warp with top_k = 3: the second group has one slot
])
def test_ragged_and_small_shapes(H, I, E, k, B):
    layer = _rand_layer_shape(H, I, E, k, seed=H + I)
    x, ids, w = workload.tokens(layer.shape, B, seed=7)
    y, h = _run_layer(layer, x, ids, w)
    y_ref, h_ref, _ = oracle.moe_layer(layer.ref, x, ids, w, return_h=True)
    _check_y(y, y_ref)
    _check_h(h, h_ref)


def test_activation_scale_extremes(q30):
    """Tokens whose activations are far from unit scale or span a wide range.

    The kernels hold activations as f16 times a per-row power of two; results
    must still match the oracle relative to the output's own scale.
    """
    B = 4
    x, ids, w = workload.tokens(q30.shape, B, batch=77)
    xf = workload.bf16_bits_to_f32(x).copy()
    xf[0] *= 1e8
    xf[1] *= 1e-8
    xf[2, ::2] *= 1e4          # half the row large, half small: range ~1e8
    xf[2, 1::2] *= 1e-4
    xf[3, :8] = [3e-9, -7e-10, 65504.0, 70000.0, -1e5, 2.0**-14, 2.0**-24, 0.0]
    xb = torch.from_numpy(xf).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    y, h = _run_layer(q30, xb, ids, w)
    y_ref, h_ref, _ = oracle.moe_layer(q30.ref, xb, ids, w, return_h=True)
    for t in range(B):
        scale = float(np.max(np.abs(y_ref[t])))
        assert scale > 0 and np.all(np.isfinite(y[t]))
        d, cos = parity_stats(y[t:t + 1] / scale, y_ref[t:t + 1] / scale)
        assert d <= 1e-4 and cos >= MIN_COS, (t, d, cos)


def test_duplicate_ids_and_all_tokens_on_one_expert(tiny):
    B = 16
    x, _, _ = workload.tokens(tiny.shape, B, batch=5)
    ids = np.full((B, 2), 3, dtype=np.int32)  # every slot -> expert 3 (duplicates within a token)
    w = np.tile(np.array([[0.75, 0.25]], np.float32), (B, 1))
    y, h = _run_layer(tiny, x, ids, w)
    y_ref, h_ref, _ = oracle.moe_layer(tiny.ref, x, ids, w, return_h=True)
    _check_y(y, y_ref)
    _check_h(h, h_ref)


def test_invalid_ids_flagged_and_skipped(tiny):
    B = 3
    x, ids, w = workload.tokens(tiny.shape, B, batch=6)
    ids = ids.copy()
    ids[0, 1] = 8      # == E
    ids[2, 0] = -5
    y, h, err = _run_layer(tiny, x, ids, w, with_err=True)
    y_ref, h_ref, bad = oracle.moe_layer(tiny.ref, x, ids, w, return_h=True)
    assert bad == 2 and err == 1
    assert np.all(h[0, 1] == 0) and np.all(h[2, 0] == 0)
    _check_y(y, y_ref)
    _check_h(h, h_ref)


@pytest.mark.parametrize("form", ["per_token", "grouped"])
@pytest.mark.parametrize("which,B,routing", [("q30", 32, "uniform"), ("q30", 64, "skewed"), ("tiny", 16, "uniform")])
def test_batch_equals_tokens_one_at_a_time(request, form, which, B, routing):
    """A token's results do not depend on the rest of the batch, for each
    moe_gate_up kernel. The per-token kernel runs a large batch with several
    slots per warp and several outputs per down warp, a single token with one
    of each, and forms every sum in the same order; the grouped kernel gives
    each pair its own MMA column. Either way results must be identical. (The
    layer entry points switch from the per-token to the grouped kernel at
    2*B*top_k >= 5E; across that switch results agree to FP32 rounding only.)"""
    layer = request.getfixturevalue(which)
    gate_up = ops.moe_gate_up if form == "per_token" else ops.moe_gate_up_grouped
    x, ids, w = workload.tokens(layer.shape, B, routing=routing, batch=500 + B)

    def run(xs, ids_, w_):
        n = xs.shape[0]
        h = torch.empty((n, layer.shape.top_k, layer.shape.I), dtype=torch.int16, device="cuda")
        y = torch.empty((n, layer.shape.H), dtype=torch.float32, device="cuda")
        idd = _dev(ids_)
        gate_up(layer.dev, _dev(xs.view(np.int16)), idd, h)
        ops.moe_down(layer.dev, h, idd, _dev(w_), y)
        torch.cuda.synchronize()
        return y.cpu().numpy(), h.cpu().numpy().view(np.uint16)

    y, h = run(x, ids, w)
    for t in range(B):
        y1, h1 = run(x[t:t + 1], ids[t:t + 1], w[t:t + 1])
        assert np.array_equal(h1[0], h[t]), t
        assert np.array_equal(y1[0], y[t]), t


def test_layer_uses_the_grouped_kernel_from_its_switch(q30):
    """moe_layer's intermediate equals moe_gate_up's below 8*B*top_k = 13E and
    moe_gate_up_grouped's from there on (Qwen-3-30B-A3B shape: 26 tokens)."""
    for B in (25, 26):
        x, ids, w = workload.tokens(q30.shape, B, batch=700 + B)
        _, h = _run_layer(q30, x, ids, w)
        hp = torch.empty((B, 8, q30.shape.I), dtype=torch.int16, device="cuda")
        hg = torch.empty_like(hp)
        ops.moe_gate_up(q30.dev, _dev(x.view(np.int16)), _dev(ids), hp)
        ops.moe_gate_up_grouped(q30.dev, _dev(x.view(np.int16)), _dev(ids), hg)
        torch.cuda.synchronize()
        grouped = 8 * B * 8 >= 13 * 128
        assert ops.layer_gate_up_kernel(q30.sh, B) == ("grouped" if grouped else "per_token")
        want = (hg if grouped else hp).cpu().numpy().view(np.uint16)
        assert np.array_equal(h, want), B


def test_invalid_ids_in_a_large_batch(tiny):
    B = 24  # several slots per gate_up warp
    x, ids, w = workload.tokens(tiny.shape, B, batch=7)
    ids = ids.copy()
    ids[3, 0] = 8
    ids[17, 1] = -1
    y, h, err = _run_layer(tiny, x, ids, w, with_err=True)
    y_ref, h_ref, bad = oracle.moe_layer(tiny.ref, x, ids, w, return_h=True)
    assert bad == 2 and err == 1
    assert np.all(h[3, 0] == 0) and np.all(h[17, 1] == 0)
    _check_y(y, y_ref)
    _check_h(h, h_ref)


def test_empty_batch_launches_nothing(tiny):
    y = torch.full((0, tiny.shape.H), 7.0, device="cuda")
    ops.moe_layer(tiny.dev, torch.empty((0, tiny.shape.H), dtype=torch.int16, device="cuda"),
                  torch.empty((0, 2), dtype=torch.int32, device="cuda"),
                  torch.empty((0, 2), dtype=torch.float32, device="cuda"),
                  torch.empty((0, 2, tiny.shape.I), dtype=torch.int16, device="cuda"), y)
    torch.cuda.synchronize()


def test_nan_scale_propagates_to_its_outputs():
    layer = _rand_layer_shape(64, 64, 2, 1, seed=3)
    # NaN E8M0 scale in down row 5 of expert 1, in both the oracle and the device copy
    layer.ref.down_scales[1, 5, 0] = 0xFF
    d_scales = layer.dev.tensors[3].view(2, 64, 2)
    d_scales[1, 5, 0] = 0xFF
    x, _, _ = workload.tokens(layer.shape, 2)
    ids = np.array([[1], [0]], np.int32)
    w = np.ones((2, 1), np.float32)
    y, _ = _run_layer(layer, x, ids, w)
    y_ref, _ = oracle.moe_layer(layer.ref, x, ids, w)
    assert np.isnan(y[0, 5]) and np.isnan(y_ref[0, 5])
    assert np.all(np.isfinite(np.delete(y[0], 5))) and np.all(np.isfinite(y[1]))


def test_deterministic_and_host_entry_point_matches(q30):
    B = 32
    x, ids, w = workload.tokens(q30.shape, B, batch=3)
    y1, h1 = _run_layer(q30, x, ids, w)
    y2, h2 = _run_layer(q30, x, ids, w)
    assert np.array_equal(y1, y2) and np.array_equal(h1, h2)
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    xh, idh, wh = pin(x.view(np.int16)), pin(ids), pin(w)
    yh = torch.empty((B, q30.shape.H), dtype=torch.float32).pin_memory()
    dev = dict(x_dev=torch.empty_like(xh, device="cuda"), ids_dev=torch.empty_like(idh, device="cuda"),
               wts_dev=torch.empty_like(wh, device="cuda"),
               h_dev=torch.empty((B, 8, q30.shape.I), dtype=torch.int16, device="cuda"),
               y_dev=torch.empty((B, q30.shape.H), dtype=torch.float32, device="cuda"))
    ops.moe_layer_host(q30.dev, xh, idh, wh, y_host=yh, **dev)
    torch.cuda.synchronize()
    assert np.array_equal(yh.numpy(), y1)


def test_library_allocates_no_device_memory(tiny):
    free0, _ = torch.cuda.mem_get_info()
    x, ids, w = workload.tokens(tiny.shape, 4)
    for _ in range(3):
        _run_layer(tiny, x, ids, w)
    free1, _ = torch.cuda.mem_get_info()
    # only torch's caching allocator may have grown (the test's own tensors)
    assert free0 - free1 < 64 << 20


def _zero_scale_layer():
    """A layer (H=256, I=256, E=2, top-1) whose gate row 5 of expert 1 keeps
    only block 0, with E8M0 scale code 0 (2^-127), and whose down row 7 of
    expert 1 likewise, in both the oracle's arrays and the device copy."""
    layer = _rand_layer_shape(256, 256, 2, 1, seed=13)
    r = layer.ref
    r.gate_codes[1, 5, 32:] = 0
    r.gate_scales[1, 5, 0] = 0
    r.down_codes[1, 7, 32:] = 0
    r.down_scales[1, 7, 0] = 0
    H, I = 256, 256
    gu_c = layer.dev.tensors[0].view(2, I, 2, H)
    gu_s = layer.dev.tensors[1].view(2, I, 2, H // 32)
    d_c = layer.dev.tensors[2].view(2, H, I)
    d_s = layer.dev.tensors[3].view(2, H, I // 32)
    gu_c[1, 5, 0, 32:] = 0
    gu_s[1, 5, 0, 0] = 0
    d_c[1, 7, 32:] = 0
    d_s[1, 7, 0] = 0
    return layer


@pytest.mark.parametrize("down_form", ["per_token", "grouped"])
def test_scale_code_zero_decodes_to_two_to_the_minus_127(down_form):
    """E8M0 code 0 is 2^-127, not 0 (the kernels decode scales with the
    hardware E8M0 -> BF16 conversion). Activations of about 2^110 make the
    one remaining block of gate row 5 give a visible g, and an intermediate of
    about 2^100 makes down row 7's block give a visible y; both rows would
    read 0 if code 0 decoded to 0."""
    layer = _zero_scale_layer()
    xf = workload.bf16_bits_to_f32(workload.tokens(layer.shape, 1, seed=3)[0]).astype(np.float64)
    xb = torch.from_numpy((xf * 2.0**110).astype(np.float32)).to(torch.bfloat16)
    x = xb.view(torch.int16).numpy().view(np.uint16)
    ids = np.array([[1]], np.int32)
    w = np.ones((1, 1), np.float32)
    _, h = _run_layer(layer, x, ids, w)
    y_ref, h_ref, _ = oracle.moe_layer(layer.ref, x, ids, w, return_h=True)
    assert _bf16_vals(h_ref[0, 0, 5:6])[0] != 0.0
    _check_h(h, h_ref)
    # down alone, from an intermediate of about 2^100
    hb = torch.from_numpy((np.linspace(-1, 1, 256) * 2.0**100).astype(np.float32)).to(torch.bfloat16)
    hbits = hb.view(torch.int16).numpy().view(np.uint16).reshape(1, 1, 256)
    y = torch.empty((1, 256), dtype=torch.float32, device="cuda")
    fn = ops.moe_down if down_form == "per_token" else ops.moe_down_grouped
    fn(layer.dev, _dev(hbits.view(np.int16)), _dev(ids), _dev(w), y)
    torch.cuda.synchronize()
    wd = oracle.dequantize_mxfp8(layer.ref.down_codes[1], layer.ref.down_scales[1])  # [H, I]
    y_exp = wd @ _bf16_vals(hbits[0, 0])
    yg = y.cpu().numpy()[0].astype(np.float64)
    assert y_exp[7] != 0.0
    rel = np.abs(yg - y_exp) / np.maximum(np.abs(y_exp), 1e-30 * 2.0**100)
    assert rel[7] <= 1e-5, (yg[7], y_exp[7])
    assert np.max(np.abs(yg - y_exp)) <= 1e-5 * np.max(np.abs(y_exp))
