"""CPU oracle for the output-centric ("warp decode") MoE decode layer.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers. The product path never
imports this package, and this package imports nothing from the product except
its seeded input generator (which the caller passes in as plain arrays).

The arithmetic lives in ``oracle.c`` (plain C, double precision,
single-threaded); this module compiles it with gcc into ``_build/`` and wraps
it for numpy arrays. Every function cites the passage it follows in the C
source.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_DIR = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_DIR, "oracle.c")
_LIB = os.path.join(_DIR, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math: IEEE double throughout)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_SRC) > os.path.getmtime(_LIB):
        tmp = _LIB + ".tmp"
        r = subprocess.run(
            ["gcc", "-O2", "-std=c11", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared",
             _SRC, "-o", tmp, "-lm"],
            capture_output=True, text=True,
        )
        if r.returncode != 0:
            raise RuntimeError("oracle build failed:\n" + r.stdout + r.stderr)
        os.replace(tmp, _LIB)
    return _LIB


def _get():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
            lib.oracle_e4m3_value.restype = ctypes.c_double
            lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
            lib.oracle_e8m0_value.restype = ctypes.c_double
            lib.oracle_e8m0_value.argtypes = [ctypes.c_uint8]
            lib.oracle_bf16_value.restype = ctypes.c_double
            lib.oracle_bf16_value.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_rne.restype = ctypes.c_uint16
            lib.oracle_bf16_rne.argtypes = [ctypes.c_double]
            lib.oracle_silu.restype = ctypes.c_double
            lib.oracle_silu.argtypes = [ctypes.c_double]
            lib.oracle_quantize_mxfp8.restype = ctypes.c_int
            lib.oracle_quantize_mxfp8.argtypes = [vp, i64, i64, vp, vp]
            lib.oracle_dequantize_mxfp8.restype = ctypes.c_int
            lib.oracle_dequantize_mxfp8.argtypes = [vp, vp, i64, i64, vp]
            lib.oracle_moe_layer.restype = i64
            lib.oracle_moe_layer.argtypes = [i32, i32, i32, i32, i32] + [vp] * 11
            lib.oracle_route.restype = ctypes.c_int
            lib.oracle_route.argtypes = [vp, i32, i32, i32, vp, vp]
            lib.oracle_moe_layer_variant.restype = i64
            lib.oracle_moe_layer_variant.argtypes = [i32, i32, i32, i32, i32] + [vp] * 9 + [i32, i32, vp]
            _lib = lib
        return _lib


def e4m3_value(code: int) -> float:
    return _get().oracle_e4m3_value(code)


def e8m0_value(s: int) -> float:
    return _get().oracle_e8m0_value(s)


def bf16_value(b: int) -> float:
    return _get().oracle_bf16_value(b)


def bf16_rne(v: float) -> int:
    return int(_get().oracle_bf16_rne(v))


def silu(g: float) -> float:
    return _get().oracle_silu(g)


def _c(a: np.ndarray, dtype) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    return a


def quantize_mxfp8(w: np.ndarray):
    """FP32 [..., K] -> (E4M3 codes uint8 [..., K], E8M0 scales uint8 [..., K/32])."""
    w = _c(w, np.float32)
    K = w.shape[-1]
    rows = w.size // K if K else 0
    codes = np.empty(w.shape, dtype=np.uint8)
    scales = np.empty(w.shape[:-1] + (K // 32,), dtype=np.uint8)
    if _get().oracle_quantize_mxfp8(w.ctypes.data, rows, K, codes.ctypes.data, scales.ctypes.data):
        raise ValueError("K must be a multiple of 32")
    return codes, scales


def dequantize_mxfp8(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    K = codes.shape[-1]
    rows = codes.size // K if K else 0
    out = np.empty(codes.shape, dtype=np.float64)
    if _get().oracle_dequantize_mxfp8(codes.ctypes.data, scales.ctypes.data, rows, K, out.ctypes.data):
        raise ValueError("K must be a multiple of 32")
    return out


class QuantizedLayer:
    """Canonical MXFP8 expert weights: gate/up [E,I,H] (+[E,I,H/32]), down [E,H,I] (+[E,H,I/32])."""

    def __init__(self, gate_codes, gate_scales, up_codes, up_scales, down_codes, down_scales):
        self.gate_codes = _c(gate_codes, np.uint8)
        self.gate_scales = _c(gate_scales, np.uint8)
        self.up_codes = _c(up_codes, np.uint8)
        self.up_scales = _c(up_scales, np.uint8)
        self.down_codes = _c(down_codes, np.uint8)
        self.down_scales = _c(down_scales, np.uint8)
        E, I, H = self.gate_codes.shape
        assert self.up_codes.shape == (E, I, H) and self.down_codes.shape == (E, H, I)
        self.E, self.I, self.H = E, I, H

    @classmethod
    def from_fp32(cls, gate: np.ndarray, up: np.ndarray, down: np.ndarray) -> "QuantizedLayer":
        gc, gs = quantize_mxfp8(gate)
        uc, us = quantize_mxfp8(up)
        dc, ds = quantize_mxfp8(down)
        return cls(gc, gs, uc, us, dc, ds)


def moe_layer(layer: QuantizedLayer, x_bits: np.ndarray, ids: np.ndarray, w: np.ndarray, return_h: bool = False):
    """FP64 MoE decode layer. Returns y [B,H] float64 (and h bits [B,k,I] uint16).

    Also returns the number of slots whose expert id is outside [0, E).
    """
    x_bits = _c(x_bits, np.uint16)
    ids = _c(ids, np.int32)
    w = _c(w, np.float32)
    B, H = x_bits.shape
    k = ids.shape[1]
    assert H == layer.H and ids.shape == (B, k) and w.shape == (B, k)
    y = np.empty((B, H), dtype=np.float64)
    h = np.empty((B, k, layer.I), dtype=np.uint16) if return_h else None
    n_bad = _get().oracle_moe_layer(
        layer.H, layer.I, layer.E, k, B,
        x_bits.ctypes.data, ids.ctypes.data, w.ctypes.data,
        layer.gate_codes.ctypes.data, layer.gate_scales.ctypes.data,
        layer.up_codes.ctypes.data, layer.up_scales.ctypes.data,
        layer.down_codes.ctypes.data, layer.down_scales.ctypes.data,
        y.ctypes.data, h.ctypes.data if h is not None else None,
    )
    if n_bad < 0:
        raise ValueError("oracle_moe_layer rejected the shape (H and I must be multiples of 32)")
    return (y, h, int(n_bad)) if return_h else (y, int(n_bad))


def moe_layer_variant(layer: QuantizedLayer, x_bits: np.ndarray, ids: np.ndarray, w: np.ndarray,
                      round_h: bool, mx_acts: bool) -> np.ndarray:
    """The layer with the intermediate rounded to BF16 or kept exact, and with or
    without an MXFP8 round trip of each projection's input activation (the
    conventional path's BF16 -> MXFP8 -> BF16). round_h=True, mx_acts=False is
    the layer itself. Returns y [B,H] float64."""
    x_bits = _c(x_bits, np.uint16)
    ids = _c(ids, np.int32)
    w = _c(w, np.float32)
    B, H = x_bits.shape
    k = ids.shape[1]
    y = np.empty((B, H), dtype=np.float64)
    n = _get().oracle_moe_layer_variant(
        layer.H, layer.I, layer.E, k, B, x_bits.ctypes.data, ids.ctypes.data, w.ctypes.data,
        layer.gate_codes.ctypes.data, layer.gate_scales.ctypes.data,
        layer.up_codes.ctypes.data, layer.up_scales.ctypes.data,
        layer.down_codes.ctypes.data, layer.down_scales.ctypes.data,
        int(round_h), int(mx_acts), y.ctypes.data)
    if n < 0:
        raise ValueError("oracle_moe_layer_variant rejected the shape")
    return y


def route(logits: np.ndarray, top_k: int):
    """Top-k routing of float32 logits [B,E]: ids int32 [B,k] (descending
    probability, ties to the lower expert index) and renormalised softmax
    weights float64 [B,k]."""
    logits = _c(logits, np.float32)
    B, E = logits.shape
    ids = np.empty((B, top_k), dtype=np.int32)
    w = np.empty((B, top_k), dtype=np.float64)
    if _get().oracle_route(logits.ctypes.data, B, E, top_k, ids.ctypes.data, w.ctypes.data):
        raise ValueError("oracle_route rejected its arguments")
    return ids, w
