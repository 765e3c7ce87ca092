"""Pins of the CPU oracle against things other than itself.

Each test checks the oracle against a library routine (torch's float8 / bf16
conversions, torch float64 matmuls), a published table, a closed form, or an
algebraic invariant of the layer, so that a dropped term, a wrong sign or
index, or a transposed operand in the oracle fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from output_centric_expert_gb300 import workload

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- decoding --

def test_e4m3_all_codes_match_torch_float8():
    """All 256 E4M3 codes: oracle value == torch.float8_e4m3fn -> float64."""
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_value(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert sorted(np.flatnonzero(nan).tolist()) == [0x7F, 0xFF]
    assert np.array_equal(ref[~nan], got[~nan])
    # sign of zero
    assert math.copysign(1.0, oracle.e4m3_value(0x80)) == -1.0


def test_e4m3_e8m0_published_table():
    """Values from the OCP MX v1.0 tables (golden fixture, cited inside)."""
    with open(os.path.join(GOLDEN, "e4m3_e8m0_table.json")) as f:
        g = json.load(f)
    for code, val in g["e4m3"]:
        v = oracle.e4m3_value(int(code, 16))
        if val == "nan":
            assert math.isnan(v)
        else:
            assert v == val and math.copysign(1.0, v) == math.copysign(1.0, val)
    for code, val in g["e8m0"]:
        v = oracle.e8m0_value(int(code, 16))
        assert math.isnan(v) if val == "nan" else v == val


def test_e8m0_all_scales_match_ldexp():
    for s in range(255):
        assert oracle.e8m0_value(s) == math.ldexp(1.0, s - 127)
    assert math.isnan(oracle.e8m0_value(255))


# -------------------------------------------------------------------- bf16 --

def test_bf16_rne_matches_torch_on_float32_values():
    """For float32-representable inputs torch's float32->bf16 cast is RNE."""
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.standard_normal(4000).astype(np.float32),
        (rng.standard_normal(2000) * 1e-30).astype(np.float32),
        (rng.standard_normal(2000) * 1e30).astype(np.float32),
        np.array([0.0, -0.0, 1.0, -1.0, 3.0e38, 1e-45, 1.00390625, 1.01171875], dtype=np.float32),
    ])
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    got = np.array([oracle.bf16_rne(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(ref, got)


def _bf16_rne_by_bits(v: float) -> int:
    """Independent RNE: round the float64 significand bits directly."""
    b = np.array([v], dtype=np.float64).view(np.uint64)[0]
    sign = int(b >> 63)
    a = abs(v)
    if a == 0.0:
        return sign << 15
    m, e = math.frexp(a)  # a = m * 2^e, m in [0.5, 1)
    # bf16 normal: 8 significant bits; below 2^-126 fixed quantum 2^-133
    q_exp = max(e - 8, -133)
    scaled = a / math.ldexp(1.0, q_exp)  # exact in double
    n = math.floor(scaled)
    frac = scaled - n
    if frac > 0.5 or (frac == 0.5 and n % 2 == 1):
        n += 1
    val = math.ldexp(n, q_exp)
    f32 = np.array([val], dtype=np.float32)
    return int(f32.view(np.uint32)[0] >> 16) | (sign << 15)


def test_bf16_rne_on_doubles_and_ties():
    rng = np.random.default_rng(2)
    vals = list(rng.standard_normal(3000)) + list(rng.standard_normal(500) * 1e-39)
    # exact ties between adjacent bf16 values (representable in double)
    for base in (1.0, 1.5, 3.0, 1e-3, 7.25):
        b16 = oracle.bf16_rne(base)
        lo, hi = oracle.bf16_value(b16), oracle.bf16_value(b16 + 1)
        vals.append((lo + hi) / 2)
        vals.append(-(lo + hi) / 2)
    for v in vals:
        assert oracle.bf16_rne(float(v)) == _bf16_rne_by_bits(float(v)), v
    # ties go to the even code
    one = oracle.bf16_rne(1.0)
    mid = (oracle.bf16_value(one) + oracle.bf16_value(one + 1)) / 2
    assert oracle.bf16_rne(mid) == one  # 0x3F80 is even
    mid2 = (oracle.bf16_value(one + 1) + oracle.bf16_value(one + 2)) / 2
    assert oracle.bf16_rne(mid2) == one + 2


def test_silu_matches_torch():
    g = torch.linspace(-40, 40, 2001, dtype=torch.float64)
    ref = torch.nn.functional.silu(g).numpy()
    got = np.array([oracle.silu(float(v)) for v in g])
    np.testing.assert_allclose(got, ref, rtol=1e-15, atol=1e-300)
    assert oracle.silu(0.0) == 0.0


# --------------------------------------------------------------- quantiser --

def _torch_mx_quantize(w: np.ndarray):
    """OCP MX v1.0 conversion with torch's float8 cast doing the rounding."""
    t = torch.from_numpy(w.astype(np.float64)).reshape(-1, 32)
    amax = t.abs().amax(dim=1)
    _, ex = torch.frexp(amax)
    s = torch.where(amax == 0, torch.zeros_like(ex), (ex - 1 - 8 + 127).clamp(0, 254))
    X = torch.pow(2.0, (s - 127).to(torch.float64))
    q = (t / X[:, None]).clamp(-448, 448).to(torch.float8_e4m3fn)
    codes = q.view(torch.uint8).reshape(w.shape).numpy()
    return codes, s.to(torch.uint8).reshape(w.shape[:-1] + (w.shape[-1] // 32,)).numpy()


def test_quantizer_matches_torch_float8_cast():
    rng = np.random.default_rng(3)
    w = (rng.standard_normal((64, 256)) * 0.05).astype(np.float32)
    w[3, :32] = 0.0  # all-zero block
    w[5, 32:64] *= 1e4  # large block
    w[7, 64:96] *= 1e-30  # tiny block
    codes, scales = oracle.quantize_mxfp8(w)
    rc, rs = _torch_mx_quantize(w)
    assert np.array_equal(scales, rs)
    assert np.array_equal(codes, rc)


def test_quantizer_roundtrip_and_error_bound():
    rng = np.random.default_rng(4)
    # exactly representable blocks survive unchanged
    exact_codes = rng.integers(0, 0x7E, size=(16, 32)).astype(np.uint8)
    exact_codes[:, 0] = 0x7E  # the block max is 448 -> scale exponent 0 after shifting
    exact_codes |= (rng.integers(0, 2, size=exact_codes.shape) << 7).astype(np.uint8)
    vals = torch.from_numpy(exact_codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    shift = rng.integers(-20, 20, size=(16, 1))
    w = (vals * np.power(2.0, shift)).astype(np.float32)
    codes, scales = oracle.quantize_mxfp8(w)
    back = oracle.dequantize_mxfp8(codes, scales)
    assert np.array_equal(back, w.astype(np.float64))
    # random blocks: relative error at most half an E4M3 ulp (2^-4) above the
    # normal range of the block, absolute error at most 2^-10 * X below it;
    # nothing exceeds the clamp
    w = (rng.standard_normal((128, 32)) * 0.05).astype(np.float32)
    codes, scales = oracle.quantize_mxfp8(w)
    back = oracle.dequantize_mxfp8(codes, scales)
    X = np.power(2.0, scales.astype(np.float64) - 127)
    err = np.abs(back - w)
    amax = np.abs(w).max(axis=1, keepdims=True)
    clipped = np.abs(w) > 448 * X
    assert np.all(back[clipped] == np.sign(w[clipped]) * 448 * np.broadcast_to(X, w.shape)[clipped])
    ok = ~clipped
    bound = np.maximum(np.abs(w) * 2.0**-4, 2.0**-10 * X)
    assert np.all(err[ok] <= bound[ok] * (1 + 1e-12))
    assert np.all(np.abs(back) <= amax * (1 + 2.0**-4))


# ------------------------------------------------------------- the layer ---

def _rand_layer(H, I, E, seed):
    rng = np.random.default_rng(seed)
    g = (rng.standard_normal((E, I, H)) * 0.05).astype(np.float32)
    u = (rng.standard_normal((E, I, H)) * 0.05).astype(np.float32)
    d = (rng.standard_normal((E, H, I)) * 0.05).astype(np.float32)
    return oracle.QuantizedLayer.from_fp32(g, u, d)


def _rand_x(B, H, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((B, H)).astype(np.float32)
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)


def _torch_dequant(codes, scales):
    v = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64)
    s = torch.pow(2.0, torch.from_numpy(scales.astype(np.float64)) - 127)
    return v * s.repeat_interleave(32, dim=-1)


def _torch_bf16_round64(t: torch.Tensor) -> torch.Tensor:
    """RNE of float64 values to bf16, via the independent bit rounding above."""
    flat = t.reshape(-1).tolist()
    bits = np.array([_bf16_rne_by_bits(v) for v in flat], dtype=np.uint16)
    return torch.from_numpy(workload.bf16_bits_to_f32(bits).astype(np.float64)).reshape(t.shape)


def _dense_reference(layer, x_bits, ids, w):
    """y = sum over ALL experts e of g_e * FFN_e(x), g_e = summed routing weight.

    A dense formulation (every expert evaluated, most with weight 0) built from
    torch float64 matmuls on torch-dequantised weights.
    """
    Wg = _torch_dequant(layer.gate_codes, layer.gate_scales)  # [E,I,H]
    Wu = _torch_dequant(layer.up_codes, layer.up_scales)
    Wd = _torch_dequant(layer.down_codes, layer.down_scales)  # [E,H,I]
    x = torch.from_numpy(workload.bf16_bits_to_f32(x_bits).astype(np.float64))  # [B,H]
    B = x.shape[0]
    gmat = torch.zeros(B, layer.E, dtype=torch.float64)
    for t in range(B):
        for j in range(ids.shape[1]):
            gmat[t, ids[t, j]] += float(w[t, j])
    y = torch.zeros(B, layer.H, dtype=torch.float64)
    for e in range(layer.E):
        gate = x @ Wg[e].T  # [B,I]
        up = x @ Wu[e].T
        h = _torch_bf16_round64(torch.nn.functional.silu(gate) * up)
        y += gmat[:, e:e + 1] * (h @ Wd[e].T)
    return y.numpy()


def test_top1_weight1_is_dense_swiglu_ffn():
    """k=1, w=1: the layer is one expert's dense SwiGLU FFN (non-square H != I)."""
    H, I, E = 64, 96, 3
    layer = _rand_layer(H, I, E, 10)
    x = _rand_x(4, H, 11)
    ids = np.array([[2], [0], [1], [2]], dtype=np.int32)
    w = np.ones((4, 1), dtype=np.float32)
    y, h, bad = oracle.moe_layer(layer, x, ids, w, return_h=True)
    assert bad == 0
    Wg = _torch_dequant(layer.gate_codes, layer.gate_scales)
    Wu = _torch_dequant(layer.up_codes, layer.up_scales)
    Wd = _torch_dequant(layer.down_codes, layer.down_scales)
    xf = torch.from_numpy(workload.bf16_bits_to_f32(x).astype(np.float64))
    for t in range(4):
        e = ids[t, 0]
        hh = _torch_bf16_round64(torch.nn.functional.silu(Wg[e] @ xf[t]) * (Wu[e] @ xf[t]))
        ref_h_bits = np.array([_bf16_rne_by_bits(v) for v in (torch.nn.functional.silu(Wg[e] @ xf[t]) * (Wu[e] @ xf[t])).tolist()], dtype=np.uint16)
        assert np.array_equal(h[t, 0], ref_h_bits)
        ref = (Wd[e] @ hh).numpy()
        np.testing.assert_allclose(y[t], ref, rtol=1e-12, atol=1e-12)


def test_brute_force_dense_formulation_tiny():
    """Tiny shapes, B=1..4: the routed (gather) oracle equals the dense all-E sum."""
    H, I, E, k = 32, 64, 5, 3
    layer = _rand_layer(H, I, E, 20)
    for B in (1, 2, 3, 4):
        x = _rand_x(B, H, 21 + B)
        rng = np.random.default_rng(30 + B)
        ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(B)]).astype(np.int32)
        w = rng.random((B, k)).astype(np.float32)
        y, bad = oracle.moe_layer(layer, x, ids, w)
        assert bad == 0
        np.testing.assert_allclose(y, _dense_reference(layer, x, ids, w), rtol=1e-12, atol=1e-12)


def test_linearity_in_routing_weights():
    H, I, E, k = 64, 32, 6, 4
    layer = _rand_layer(H, I, E, 40)
    x = _rand_x(3, H, 41)
    rng = np.random.default_rng(42)
    ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(3)]).astype(np.int32)
    # dyadic weights so that alpha*w1 + beta*w2 is exact in float32
    w1 = (rng.integers(0, 64, size=(3, k)) / 64.0).astype(np.float32)
    w2 = (rng.integers(0, 64, size=(3, k)) / 64.0).astype(np.float32)
    a, b = 0.75, -2.5
    y1, _ = oracle.moe_layer(layer, x, ids, w1)
    y2, _ = oracle.moe_layer(layer, x, ids, w2)
    y12, _ = oracle.moe_layer(layer, x, ids, (a * w1 + b * w2).astype(np.float32))
    np.testing.assert_allclose(y12, a * y1 + b * y2, rtol=1e-12, atol=1e-12)
    # y is the sum of its single-slot results
    parts = sum(oracle.moe_layer(layer, x, ids[:, j:j + 1], w1[:, j:j + 1])[0] for j in range(k))
    np.testing.assert_allclose(y1, parts, rtol=1e-12, atol=1e-12)


def test_slot_permutation_invariance_and_duplicates():
    H, I, E, k = 32, 32, 4, 4
    layer = _rand_layer(H, I, E, 50)
    x = _rand_x(2, H, 51)
    ids = np.array([[3, 0, 2, 1], [1, 1, 2, 0]], dtype=np.int32)  # token 1 repeats expert 1
    w = np.array([[0.4, 0.3, 0.2, 0.1], [0.25, 0.5, 0.125, 0.125]], dtype=np.float32)
    y, _ = oracle.moe_layer(layer, x, ids, w)
    perm = [2, 0, 3, 1]
    yp, _ = oracle.moe_layer(layer, x, ids[:, perm], w[:, perm])
    np.testing.assert_allclose(yp, y, rtol=1e-12, atol=1e-12)
    # duplicate ids add: token 1's two slots on expert 1 == one slot of weight 0.75
    ymerged, _ = oracle.moe_layer(layer, x[1:], np.array([[1, 2, 0]], dtype=np.int32),
                                  np.array([[0.75, 0.125, 0.125]], dtype=np.float32))
    np.testing.assert_allclose(y[1:], ymerged, rtol=1e-12, atol=1e-12)


def _const_layer(H, I, E, gate_code, up_code, down_code, scale=127):
    gc = np.full((E, I, H), gate_code, np.uint8)
    uc = np.full((E, I, H), up_code, np.uint8)
    dc = np.full((E, H, I), down_code, np.uint8)
    return oracle.QuantizedLayer(gc, np.full((E, I, H // 32), scale, np.uint8),
                                 uc, np.full((E, I, H // 32), scale, np.uint8),
                                 dc, np.full((E, H, I // 32), scale, np.uint8))


def test_closed_form_constant_weights():
    """Constant codes: g = cg*sum(x), u = cu*sum(x), y = w*cd*I*bf16(silu(g)*u).

    Gate = -1, up = +1 separates gate from up (a swap changes the result by
    ~10^13), and scale 128 (= 2) checks the scale is applied per element.
    """
    H, I, E = 32, 64, 2
    one = np.float32(1.0)
    x = np.full((1, H), 0x3F80, dtype=np.uint16)  # bf16 1.0
    # gate code -1.0 (0xB8), up +1.0 (0x38), down 0.5 (0x30), all scales 2^(128-127) = 2
    layer = _const_layer(H, I, E, 0xB8, 0x38, 0x30, scale=128)
    ids = np.array([[1]], dtype=np.int32)
    w = np.array([[one]], dtype=np.float32)
    y, h, _ = oracle.moe_layer(layer, x, ids, w, return_h=True)
    g, u = -2.0 * H, 2.0 * H
    hv = g / (1 + math.exp(-g)) * u
    hb = _bf16_rne_by_bits(hv)
    assert np.all(h == hb)
    hval = float(workload.bf16_bits_to_f32(np.array([hb], np.uint16))[0])
    np.testing.assert_allclose(y, np.full((1, H), 1.0 * I * hval), rtol=1e-14)
    # swapped gate/up would give silu(+64)*(-64) = -4096
    assert abs(hval) < 1e-20
    # positive gate: h = bf16(silu(64)*64) ~ 4096, y = 0.5*2*I*h per output
    layer2 = _const_layer(H, I, E, 0x38, 0x38, 0x30, scale=128)
    w2 = np.array([[0.5]], dtype=np.float32)
    y2, h2, _ = oracle.moe_layer(layer2, x, ids, w2, return_h=True)
    g2 = 2.0 * H
    hb2 = _bf16_rne_by_bits(g2 / (1 + math.exp(-g2)) * g2)
    h2val = float(workload.bf16_bits_to_f32(np.array([hb2], np.uint16))[0])
    assert np.all(h2 == hb2)
    np.testing.assert_allclose(y2, np.full((1, H), 0.5 * I * h2val), rtol=1e-14)


def test_invalid_ids_contribute_nothing():
    H, I, E, k = 32, 32, 3, 2
    layer = _rand_layer(H, I, E, 60)
    x = _rand_x(2, H, 61)
    ids = np.array([[1, 7], [-1, 2]], dtype=np.int32)
    w = np.array([[0.5, 0.5], [0.5, 0.5]], dtype=np.float32)
    y, h, bad = oracle.moe_layer(layer, x, ids, w, return_h=True)
    assert bad == 2
    assert np.all(h[0, 1] == 0) and np.all(h[1, 0] == 0)
    y_ok0, _ = oracle.moe_layer(layer, x[:1], ids[:1, :1], w[:1, :1])
    y_ok1, _ = oracle.moe_layer(layer, x[1:], ids[1:, 1:], w[1:, 1:])
    np.testing.assert_allclose(y, np.concatenate([y_ok0, y_ok1]), rtol=0, atol=0)


def test_empty_batch():
    layer = _rand_layer(32, 32, 2, 70)
    y, bad = oracle.moe_layer(layer, np.zeros((0, 32), np.uint16), np.zeros((0, 1), np.int32),
                              np.zeros((0, 1), np.float32))
    assert y.shape == (0, 32) and bad == 0


def test_nan_code_propagates():
    H, I, E = 32, 32, 1
    layer = _rand_layer(H, I, E, 80)
    layer.down_codes[0, 5, 7] = 0x7F  # NaN element in output row 5
    x = _rand_x(1, H, 81)
    y, _ = oracle.moe_layer(layer, x, np.array([[0]], np.int32), np.array([[1.0]], np.float32))
    assert np.isnan(y[0, 5]) and np.all(np.isfinite(np.delete(y[0], 5)))


def test_buffer_arithmetic_from_the_pages():
    """The per-token per-expert output buffer the method removes: k*H*2 bytes."""
    with open(os.path.join(GOLDEN, "paper_figures.json")) as f:
        g = json.load(f)["per_token_intermediate_buffer_bytes"]
    q30 = workload.SHAPES["q30"]
    assert q30.top_k == g["experts"] and q30.H == g["hidden"]
    assert q30.top_k * q30.H * g["bytes_per_element"] == g["value"] == 32 * 1024


# ------------------------------------------------------------------ router --

def test_router_matches_torch_softmax_topk():
    """Distinct logits: oracle.route == torch softmax (float64) + topk + renorm."""
    rng = np.random.default_rng(7)
    L = rng.standard_normal((20, 64)).astype(np.float32)
    ids, w = oracle.route(L, 6)
    p = torch.softmax(torch.from_numpy(L.astype(np.float64)), dim=1)
    pv, pi = torch.topk(p, 6, dim=1)
    assert np.array_equal(ids, pi.numpy().astype(np.int32))
    np.testing.assert_allclose(w, (pv / pv.sum(dim=1, keepdim=True)).numpy(), rtol=1e-14)


def test_router_ties_and_special_cases():
    L = np.array([[1.0, 3.0, 3.0, 0.5, 3.0]], np.float32)
    ids, w = oracle.route(L, 3)
    assert ids.tolist() == [[1, 2, 4]]  # equal logits: lower index first
    np.testing.assert_allclose(w, [[1 / 3, 1 / 3, 1 / 3]], rtol=1e-15)
    ids, w = oracle.route(L, 1)  # top-1: weight exactly 1
    assert ids.tolist() == [[1]] and w.tolist() == [[1.0]]
    ids, w = oracle.route(np.zeros((1, 4), np.float32), 4)  # k = E, all equal
    assert ids.tolist() == [[0, 1, 2, 3]] and np.allclose(w, 0.25)
