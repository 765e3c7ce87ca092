"""Seeded synthetic workloads for the decode-time MoE layer.

Inputs only -- this module holds none of the layer's arithmetic. It is shared by
the CUDA path's tests/benchmark and by the CPU oracle's tests.

Shapes are the "Qwen-3-style" MoE layers the warp-decode pages benchmark
("Better MoE model inference with warp decode", Key claims
[§End-to-end decode throughput at scale]; the 8 x 2048 x 2 B intermediate of
[§Buffer elimination] fixes top-8 and hidden 2048), plus a tiny layer and a
larger 235B-style layer. Values:

* x  ~ N(0, 1), drawn in double and rounded to float then BF16 (RNE);
* W_gate, W_up ``[E, I, H]`` and W_down ``[E, H, I]`` ~ N(0, 0.05^2) in FP32
  (quantised to MXFP8 later, by the product packer or the oracle's quantiser);
* routing: logits ~ N(0, 1) per (token, expert), plus for "skewed" routing a
  per-expert bias with variance 2 (std sqrt(2)) shared by all tokens; softmax
  over E, top-k, renormalised to sum 1.

Every tensor is its own counter-based splitmix64 stream keyed by
(seed, stream id), so experts can be generated one at a time and in parallel.
"""
from __future__ import annotations

import ctypes
import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np

from . import _native

WEIGHT_STD = 0.05
SKEW_BIAS_STD = math.sqrt(2.0)

# stream ids (see module docstring); layer/batch indices are folded in below
_STREAM_X, _STREAM_LOGITS, _STREAM_BIAS = 1, 2, 3
_STREAM_GATE, _STREAM_UP, _STREAM_DOWN = 16, 17, 18


@dataclass(frozen=True)
class LayerShape:
    """MoE layer shape: hidden H, intermediate I, experts E, experts per token."""

    H: int
    I: int
    E: int
    top_k: int

    def expert_weight_elems(self) -> int:
        return 3 * self.H * self.I


SHAPES = {
    "tiny": LayerShape(256, 128, 8, 2),
    "q30": LayerShape(2048, 768, 128, 8),  # Qwen-3-30B-A3B-shaped layer
    "q235": LayerShape(4096, 1536, 128, 8),  # Qwen-3-235B-A22B-shaped layer
    # shape variants ("Better MoE model inference with warp decode", Why it's
    # interesting: does the flip carry over to fine-grained MoE such as
    # DeepSeek-V3?): routed experts only, by shape
    "dsv3": LayerShape(7168, 2048, 256, 8),  # DeepSeek-V3-shaped routed-expert layer
    "mixtral": LayerShape(4096, 14336, 8, 2),  # Mixtral-8x7B-shaped layer (few, wide experts)
}


@dataclass(frozen=True)
class Workload:
    """One named configuration: a layer shape, a batch size and a routing law."""

    name: str
    shape: LayerShape
    B: int
    routing: str = "uniform"  # "uniform" | "skewed"
    seed: int = 0


def _sweep():
    out = {}
    for r in ("uniform", "skewed"):
        for b in (1, 2, 4, 8, 16, 32, 64):
            out[f"q30_{r}_b{b}"] = Workload(f"q30_{r}_b{b}", SHAPES["q30"], b, r)
    return out


WORKLOADS: dict[str, Workload] = {
    "tiny_b1": Workload("tiny_b1", SHAPES["tiny"], 1),
    "q30_b1": Workload("q30_b1", SHAPES["q30"], 1),
    "q30_b32": Workload("q30_b32", SHAPES["q30"], 32),
    **_sweep(),
    **{f"q235_b{b}": Workload(f"q235_b{b}", SHAPES["q235"], b) for b in (1, 16, 64)},
    **{f"dsv3_b{b}": Workload(f"dsv3_b{b}", SHAPES["dsv3"], b) for b in (1, 16, 64)},
    **{f"mixtral_b{b}": Workload(f"mixtral_b{b}", SHAPES["mixtral"], b) for b in (1, 16, 64)},
    # batches between the listed ones, for measuring where the layer's kernel
    # choices should switch
    **{f"q235_b{b}": Workload(f"q235_b{b}", SHAPES["q235"], b) for b in (8, 12, 20, 24, 32, 40, 48)},
    **{f"dsv3_b{b}": Workload(f"dsv3_b{b}", SHAPES["dsv3"], b) for b in (24, 32, 48)},
    **{f"mixtral_b{b}": Workload(f"mixtral_b{b}", SHAPES["mixtral"], b) for b in (2, 4, 8)},
    **{f"q30_uniform_b{b}": Workload(f"q30_uniform_b{b}", SHAPES["q30"], b) for b in (24, 40, 48, 56)},
}


def _lib() -> ctypes.CDLL:
    lib = _native.load(_native.build_workload)
    if not getattr(lib, "_wl_typed", False):
        u64, i32 = ctypes.c_uint64, ctypes.c_int32
        lib.wl_splitmix64_at.restype = u64
        lib.wl_splitmix64_at.argtypes = [u64, u64]
        lib.wl_stream_key.restype = u64
        lib.wl_stream_key.argtypes = [u64, u64]
        lib.wl_normal_at.restype = ctypes.c_double
        lib.wl_normal_at.argtypes = [u64, u64]
        lib.wl_normal_f32.restype = None
        lib.wl_normal_f32.argtypes = [u64, u64, u64, ctypes.c_double, ctypes.c_double, ctypes.c_void_p]
        lib.wl_normal_bf16.restype = None
        lib.wl_normal_bf16.argtypes = [u64, u64, u64, ctypes.c_void_p]
        lib.wl_logits.restype = None
        lib.wl_logits.argtypes = [u64, u64, ctypes.c_double, i32, i32, ctypes.c_void_p]
        lib.wl_route.restype = ctypes.c_int
        lib.wl_route.argtypes = [u64, u64, ctypes.c_double, i32, i32, i32, ctypes.c_void_p, ctypes.c_void_p]
        lib._wl_typed = True
    return lib


def splitmix64_at(key: int, i: int) -> int:
    return int(_lib().wl_splitmix64_at(key, i))


def stream_key(seed: int, stream: int) -> int:
    return int(_lib().wl_stream_key(seed, stream))


def normal_f32(key: int, start: int, count: int, std: float = 1.0) -> np.ndarray:
    out = np.empty(count, dtype=np.float32)
    _lib().wl_normal_f32(key, start, count, 0.0, std, out.ctypes.data)
    return out


def _weight_stream(kind: int, layer: int) -> int:
    return kind + 64 * layer


def _token_stream(kind: int, batch: int) -> int:
    return kind + 64 * (batch + 1) * 4096


def expert_weights(shape: LayerShape, e: int, seed: int = 0, layer: int = 0):
    """FP32 weights of expert e: gate [I,H], up [I,H], down [H,I]."""
    H, I = shape.H, shape.I
    lib = _lib()
    out = []
    for kind, rows, cols in ((_STREAM_GATE, I, H), (_STREAM_UP, I, H), (_STREAM_DOWN, H, I)):
        key = lib.wl_stream_key(seed, _weight_stream(kind, layer))
        a = np.empty((rows, cols), dtype=np.float32)
        lib.wl_normal_f32(key, e * rows * cols, rows * cols, 0.0, WEIGHT_STD, a.ctypes.data)
        out.append(a)
    return tuple(out)


def all_weights(shape: LayerShape, seed: int = 0, layer: int = 0, experts=None, threads: int | None = None):
    """FP32 weights of all (or the listed) experts: gate/up [n,I,H], down [n,H,I]."""
    experts = list(range(shape.E)) if experts is None else list(experts)
    n = len(experts)
    gate = np.empty((n, shape.I, shape.H), dtype=np.float32)
    up = np.empty_like(gate)
    down = np.empty((n, shape.H, shape.I), dtype=np.float32)

    def one(idx):
        g, u, d = expert_weights(shape, experts[idx], seed, layer)
        gate[idx], up[idx], down[idx] = g, u, d

    threads = threads or min(16, os.cpu_count() or 1)
    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(one, range(n)))
    return gate, up, down


def tokens(shape: LayerShape, B: int, seed: int = 0, batch: int = 0, routing: str = "uniform"):
    """Decode-step inputs: x BF16 bits uint16 [B,H], ids int32 [B,k], weights f32 [B,k]."""
    if routing not in ("uniform", "skewed"):
        raise ValueError(f"unknown routing {routing!r}")
    lib = _lib()
    x = np.empty((B, shape.H), dtype=np.uint16)
    if B:
        lib.wl_normal_bf16(lib.wl_stream_key(seed, _token_stream(_STREAM_X, batch)), 0, B * shape.H, x.ctypes.data)
    ids = np.empty((B, shape.top_k), dtype=np.int32)
    w = np.empty((B, shape.top_k), dtype=np.float32)
    bias_std = SKEW_BIAS_STD if routing == "skewed" else 0.0
    rc = lib.wl_route(
        lib.wl_stream_key(seed, _token_stream(_STREAM_LOGITS, batch)),
        lib.wl_stream_key(seed, _weight_stream(_STREAM_BIAS, 0)),
        bias_std, B, shape.E, shape.top_k, ids.ctypes.data, w.ctypes.data,
    )
    if rc != 0:
        raise ValueError("wl_route rejected its arguments")
    return x, ids, w


def logits(shape: LayerShape, B: int, seed: int = 0, batch: int = 0, routing: str = "uniform"):
    """The router logits of the same decode step as tokens(), as float32 [B,E]
    (for a router that runs on the device instead of in the generator)."""
    if routing not in ("uniform", "skewed"):
        raise ValueError(f"unknown routing {routing!r}")
    lib = _lib()
    out = np.empty((B, shape.E), dtype=np.float32)
    if B:
        lib.wl_logits(lib.wl_stream_key(seed, _token_stream(_STREAM_LOGITS, batch)),
                      lib.wl_stream_key(seed, _weight_stream(_STREAM_BIAS, 0)),
                      SKEW_BIAS_STD if routing == "skewed" else 0.0, B, shape.E, out.ctypes.data)
    return out


def bf16_bits_to_f32(x_bits: np.ndarray) -> np.ndarray:
    """Reinterpret BF16 bit patterns as float32 values (exact widening)."""
    return (x_bits.astype(np.uint32) << 16).view(np.float32)
