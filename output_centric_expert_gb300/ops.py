"""Thin Python binding of ``libwarp_decode.so`` (argument marshalling only).

Every function here has the name of the C entry point it calls
(``include/warp_decode.h``) and does nothing but check tensor metadata,
extract pointers and raise on a non-OK status. All arithmetic of the layer runs
in the CUDA kernels (and the packer's quantisation in the library's host code).
PyTorch provides device memory and streams only. There is no fallback: if the
library cannot be built or loaded, or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import numpy as np
import torch

from . import _native

MOE_OK = 0
GU_CODES, GU_SCALES, D_CODES, D_SCALES = 0, 1, 2, 3


class MoeShape(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int32), ("I", ctypes.c_int32), ("E", ctypes.c_int32),
                ("top_k", ctypes.c_int32)]


class MoeWeights(ctypes.Structure):
    _fields_ = [("gu_codes", ctypes.c_void_p), ("gu_scales", ctypes.c_void_p),
                ("d_codes", ctypes.c_void_p), ("d_scales", ctypes.c_void_p)]


class WarpDecodeError(RuntimeError):
    def __init__(self, fn: str, status: int, detail: str):
        super().__init__(f"{fn} failed: status {status} ({status_string(status)}) {detail}".rstrip())
        self.status = status


_lib_cache = None


def lib() -> ctypes.CDLL:
    """The loaded C-ABI library (built on first use; raises if unavailable)."""
    global _lib_cache
    if _lib_cache is None:
        L = _native.load(_native.build_warp_decode)
        vp, i32, sp = ctypes.c_void_p, ctypes.c_int32, ctypes.POINTER(MoeShape)
        wp = ctypes.POINTER(MoeWeights)
        L.moe_packed_bytes.restype = ctypes.c_size_t
        L.moe_packed_bytes.argtypes = [sp, ctypes.c_int]
        L.moe_pack_weights.restype = ctypes.c_int
        L.moe_pack_weights.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp]
        L.moe_gate_up.restype = ctypes.c_int
        L.moe_gate_up.argtypes = [sp, wp, vp, vp, i32, vp, vp, vp]
        L.moe_gate_up_grouped.restype = ctypes.c_int
        L.moe_gate_up_grouped.argtypes = [sp, wp, vp, vp, i32, vp, vp, vp]
        L.moe_layer_gate_up_kernel.restype = ctypes.c_int
        L.moe_layer_gate_up_kernel.argtypes = [sp, wp, i32, ctypes.POINTER(ctypes.c_int32)]
        L.moe_down.restype = ctypes.c_int
        L.moe_down.argtypes = [sp, wp, vp, vp, vp, i32, vp, vp, vp]
        L.moe_down_grouped.restype = ctypes.c_int
        L.moe_down_grouped.argtypes = [sp, wp, vp, vp, vp, i32, vp, vp, vp]
        L.moe_layer_down_kernel.restype = ctypes.c_int
        L.moe_layer_down_kernel.argtypes = [sp, wp, i32, ctypes.POINTER(ctypes.c_int32)]
        L.moe_layer_host_kernels.restype = ctypes.c_int
        L.moe_layer_host_kernels.argtypes = [sp, wp, vp, i32, ctypes.POINTER(ctypes.c_int32),
                                             ctypes.POINTER(ctypes.c_int32)]
        L.moe_layer.restype = ctypes.c_int
        L.moe_layer.argtypes = [sp, wp, vp, vp, vp, i32, vp, vp, vp, vp]
        L.moe_route.restype = ctypes.c_int
        L.moe_route.argtypes = [sp, vp, i32, vp, vp, vp]
        L.moe_layer_routed.restype = ctypes.c_int
        L.moe_layer_routed.argtypes = [sp, wp, vp, vp, i32, vp, vp, vp, vp, vp, vp]
        L.moe_layer_noalloc.restype = ctypes.c_int
        L.moe_layer_noalloc.argtypes = [sp, wp, vp, vp, vp, i32, vp, vp, vp]
        L.moe_layer_host.restype = ctypes.c_int
        L.moe_layer_host.argtypes = [sp, wp, vp, vp, vp, i32, vp, vp, vp, vp, vp, vp, vp, vp]
        L.moe_local_ids.restype = ctypes.c_int
        L.moe_local_ids.argtypes = [sp, vp, i32, i32, i32, vp, vp, vp]
        L.moe_status_string.restype = ctypes.c_char_p
        L.moe_status_string.argtypes = [ctypes.c_int]
        L.moe_last_error.restype = ctypes.c_char_p
        L.moe_last_error.argtypes = []
        _lib_cache = L
    return _lib_cache


def status_string(status: int) -> str:
    return lib().moe_status_string(status).decode()


def _check(fn: str, status: int) -> None:
    if status != MOE_OK:
        raise WarpDecodeError(fn, status, lib().moe_last_error().decode())


def make_shape(H: int, I: int, E: int, top_k: int) -> MoeShape:
    return MoeShape(H, I, E, top_k)


def moe_packed_bytes(shape: MoeShape, which: int) -> int:
    return int(lib().moe_packed_bytes(ctypes.byref(shape), which))


@dataclass
class PackedHost:
    """Packed MXFP8 weights in host memory (numpy uint8), layout of warp_decode.h."""

    gu_codes: np.ndarray
    gu_scales: np.ndarray
    d_codes: np.ndarray
    d_scales: np.ndarray


def empty_packed_host(shape: MoeShape) -> PackedHost:
    return PackedHost(*(np.empty(moe_packed_bytes(shape, w), dtype=np.uint8) for w in range(4)))


def moe_pack_weights(shape: MoeShape, w_gate: np.ndarray, w_up: np.ndarray, w_down: np.ndarray,
                     out: PackedHost | None = None, expert_offset: int = 0) -> PackedHost:
    """Quantise FP32 weights ([E,I,H], [E,I,H], [E,H,I]) into the packed layout.

    With ``out`` and ``expert_offset``, the given experts are packed into the
    matching slices of a larger buffer (the arrays then hold len(w_gate) experts).
    """
    n = w_gate.shape[0]
    for a, shp in ((w_gate, (n, shape.I, shape.H)), (w_up, (n, shape.I, shape.H)),
                   (w_down, (n, shape.H, shape.I))):
        if a.dtype != np.float32 or a.shape != shp or not a.flags.c_contiguous:
            raise ValueError(f"expected contiguous float32 {shp}, got {a.dtype} {a.shape}")
    sub = MoeShape(shape.H, shape.I, n, min(shape.top_k, n))
    out = out or empty_packed_host(MoeShape(shape.H, shape.I, n, sub.top_k))
    per = [moe_packed_bytes(sub, w) for w in range(4)]
    arrs = [out.gu_codes, out.gu_scales, out.d_codes, out.d_scales]
    ptrs = []
    for a, nb in zip(arrs, per):
        start = expert_offset * nb
        if a.dtype != np.uint8 or a.size < start + nb or not a.flags.c_contiguous:
            raise ValueError("packed output buffer too small or not contiguous uint8")
        ptrs.append(a.ctypes.data + start)
    _check("moe_pack_weights", lib().moe_pack_weights(
        ctypes.byref(sub), w_gate.ctypes.data, w_up.ctypes.data, w_down.ctypes.data, *ptrs))
    return out


class DeviceWeights:
    """Packed MXFP8 weights resident on the GPU (four torch uint8 tensors)."""

    def __init__(self, shape: MoeShape, packed: PackedHost, device="cuda"):
        self.shape = shape
        self.tensors = [torch.from_numpy(a).to(device) for a in
                        (packed.gu_codes, packed.gu_scales, packed.d_codes, packed.d_scales)]
        for t, w in zip(self.tensors, range(4)):
            if t.numel() != moe_packed_bytes(shape, w):
                raise ValueError("packed array size does not match the shape")
        self.struct = MoeWeights(*(t.data_ptr() for t in self.tensors))

    @property
    def nbytes(self) -> int:
        return sum(t.numel() for t in self.tensors)


def _ptr(t: torch.Tensor | None, dtypes, name: str) -> int | None:
    if t is None:
        return None
    if t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype} not in {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    return t.data_ptr()


_BF16 = (torch.bfloat16, torch.int16, torch.uint16) if hasattr(torch, "uint16") else (torch.bfloat16, torch.int16)


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def moe_gate_up(weights: DeviceWeights, x: torch.Tensor, ids: torch.Tensor, h: torch.Tensor,
                err_flag: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """h[B,k,I] (bf16) = bf16(silu(x Wg^T) * (x Wu^T)) per routed slot."""
    B = x.shape[0]
    _check("moe_gate_up", lib().moe_gate_up(
        ctypes.byref(weights.shape), ctypes.byref(weights.struct), _ptr(x, _BF16, "x"),
        _ptr(ids, (torch.int32,), "ids"), B, _ptr(h, _BF16, "h"),
        _ptr(err_flag, (torch.int32,), "err_flag"), _stream(stream)))
    return h


def moe_gate_up_grouped(weights: DeviceWeights, x: torch.Tensor, ids: torch.Tensor,
                        h: torch.Tensor, err_flag: torch.Tensor | None = None,
                        stream=None) -> torch.Tensor:
    """moe_gate_up by the expert-grouped kernel (tensor-core MMAs over the pairs
    routed to each expert); same result up to FP32 rounding order."""
    B = x.shape[0]
    _check("moe_gate_up_grouped", lib().moe_gate_up_grouped(
        ctypes.byref(weights.shape), ctypes.byref(weights.struct), _ptr(x, _BF16, "x"),
        _ptr(ids, (torch.int32,), "ids"), B, _ptr(h, _BF16, "h"),
        _ptr(err_flag, (torch.int32,), "err_flag"), _stream(stream)))
    return h


def layer_gate_up_kernel(shape: MoeShape, B: int, weights: "DeviceWeights | None" = None) -> str:
    """The gate/up kernel the layer entry points run at batch B, as the library
    reports it (moe_layer_gate_up_kernel): "per_token" (moe_gate_up's) or
    "grouped" (moe_gate_up_grouped's). Without `weights` the scales are taken
    to be aligned, as DeviceWeights allocates them."""
    out = ctypes.c_int32(-1)
    _check("moe_layer_gate_up_kernel", lib().moe_layer_gate_up_kernel(
        ctypes.byref(shape), ctypes.byref(weights.struct) if weights is not None else None, B,
        ctypes.byref(out)))
    return "grouped" if out.value == 1 else "per_token"


def moe_down(weights: DeviceWeights, h: torch.Tensor, ids: torch.Tensor, wts: torch.Tensor,
             y: torch.Tensor, err_flag: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y[B,H] (fp32) = sum_j wts[:,j] * (h[:,j] Wd[ids[:,j]]^T)."""
    B = ids.shape[0]
    _check("moe_down", lib().moe_down(
        ctypes.byref(weights.shape), ctypes.byref(weights.struct), _ptr(h, _BF16, "h"),
        _ptr(ids, (torch.int32,), "ids"), _ptr(wts, (torch.float32,), "wts"), B,
        _ptr(y, (torch.float32,), "y"), _ptr(err_flag, (torch.int32,), "err_flag"),
        _stream(stream)))
    return y


def moe_down_grouped(weights: DeviceWeights, h: torch.Tensor, ids: torch.Tensor,
                     wts: torch.Tensor, y: torch.Tensor, err_flag: torch.Tensor | None = None,
                     stream=None) -> torch.Tensor:
    """moe_down by the expert-grouped kernel (each down weight decoded once,
    tensor-core MMAs over the pairs routed to each expert); same result up to
    FP32 rounding order."""
    B = ids.shape[0]
    _check("moe_down_grouped", lib().moe_down_grouped(
        ctypes.byref(weights.shape), ctypes.byref(weights.struct), _ptr(h, _BF16, "h"),
        _ptr(ids, (torch.int32,), "ids"), _ptr(wts, (torch.float32,), "wts"), B,
        _ptr(y, (torch.float32,), "y"), _ptr(err_flag, (torch.int32,), "err_flag"),
        _stream(stream)))
    return y


def layer_down_kernel(shape: MoeShape, B: int, weights: "DeviceWeights | None" = None) -> str:
    """The down kernel the layer entry points run at batch B, as the library
    reports it (moe_layer_down_kernel): "per_token" or "grouped"."""
    out = ctypes.c_int32(-1)
    _check("moe_layer_down_kernel", lib().moe_layer_down_kernel(
        ctypes.byref(shape), ctypes.byref(weights.struct) if weights is not None else None, B,
        ctypes.byref(out)))
    return "grouped" if out.value == 1 else "per_token"


def layer_host_kernels(shape: MoeShape, ids_host: np.ndarray,
                       weights: "DeviceWeights | None" = None) -> tuple[str, str]:
    """The (gate/up, down) kernels moe_layer_host runs for a batch whose ids are
    given on the host (moe_layer_host_kernels): each "per_token" or "grouped"."""
    ids_host = np.ascontiguousarray(ids_host, dtype=np.int32)
    B = ids_host.shape[0] if ids_host.ndim else 0
    gu, dn = ctypes.c_int32(-1), ctypes.c_int32(-1)
    _check("moe_layer_host_kernels", lib().moe_layer_host_kernels(
        ctypes.byref(shape), ctypes.byref(weights.struct) if weights is not None else None,
        ids_host.ctypes.data_as(ctypes.c_void_p), B, ctypes.byref(gu), ctypes.byref(dn)))
    name = {0: "per_token", 1: "grouped"}
    return name[gu.value], name[dn.value]


def moe_layer(weights: DeviceWeights, x: torch.Tensor, ids: torch.Tensor, wts: torch.Tensor,
              h_scratch: torch.Tensor, y: torch.Tensor, err_flag: torch.Tensor | None = None,
              stream=None) -> torch.Tensor:
    """The whole layer (both kernels) on the stream; returns y."""
    B = x.shape[0]
    _check("moe_layer", lib().moe_layer(
        ctypes.byref(weights.shape), ctypes.byref(weights.struct), _ptr(x, _BF16, "x"),
        _ptr(ids, (torch.int32,), "ids"), _ptr(wts, (torch.float32,), "wts"), B,
        _ptr(h_scratch, _BF16, "h_scratch"), _ptr(y, (torch.float32,), "y"),
        _ptr(err_flag, (torch.int32,), "err_flag"), _stream(stream)))
    return y


def moe_route(shape: MoeShape, logits: torch.Tensor, ids: torch.Tensor, wts: torch.Tensor,
              stream=None):
    """ids[B,k], wts[B,k] = top-k routing of FP32 logits [B,E] (on the device)."""
    B = logits.shape[0]
    _check("moe_route", lib().moe_route(
        ctypes.byref(shape), _ptr(logits, (torch.float32,), "logits"), B,
        _ptr(ids, (torch.int32,), "ids"), _ptr(wts, (torch.float32,), "wts"), _stream(stream)))
    return ids, wts


def moe_layer_routed(weights: DeviceWeights, x: torch.Tensor, logits: torch.Tensor,
                     h_scratch: torch.Tensor, y: torch.Tensor, ids_out: torch.Tensor | None = None,
                     wts_out: torch.Tensor | None = None, err_flag: torch.Tensor | None = None,
                     stream=None) -> torch.Tensor:
    """The layer from router logits (both kernels route each token themselves)."""
    B = x.shape[0]
    _check("moe_layer_routed", lib().moe_layer_routed(
        ctypes.byref(weights.shape), ctypes.byref(weights.struct), _ptr(x, _BF16, "x"),
        _ptr(logits, (torch.float32,), "logits"), B, _ptr(h_scratch, _BF16, "h_scratch"),
        _ptr(y, (torch.float32,), "y"), _ptr(ids_out, (torch.int32,), "ids_out"),
        _ptr(wts_out, (torch.float32,), "wts_out"), _ptr(err_flag, (torch.int32,), "err_flag"),
        _stream(stream)))
    return y


def moe_layer_noalloc(weights: DeviceWeights, x: torch.Tensor, ids: torch.Tensor,
                      wts: torch.Tensor, y: torch.Tensor, err_flag: torch.Tensor | None = None,
                      stream=None) -> torch.Tensor:
    """The whole layer without a caller-provided intermediate buffer.

    For callers that cannot allocate device memory: the intermediate lives in
    a fixed array inside the library (at most MOE_NOALLOC_MAX_INTERMEDIATE
    BF16 values, B * top_k * I), shared by all calls.
    """
    B = x.shape[0]
    _check("moe_layer_noalloc", lib().moe_layer_noalloc(
        ctypes.byref(weights.shape), ctypes.byref(weights.struct), _ptr(x, _BF16, "x"),
        _ptr(ids, (torch.int32,), "ids"), _ptr(wts, (torch.float32,), "wts"), B,
        _ptr(y, (torch.float32,), "y"), _ptr(err_flag, (torch.int32,), "err_flag"),
        _stream(stream)))
    return y


MOE_NOALLOC_MAX_INTERMEDIATE = 1 << 20


def moe_layer_host(weights: DeviceWeights, x_host: torch.Tensor, ids_host: torch.Tensor,
                   wts_host: torch.Tensor, x_dev: torch.Tensor, ids_dev: torch.Tensor,
                   wts_dev: torch.Tensor, h_dev: torch.Tensor, y_dev: torch.Tensor,
                   y_host: torch.Tensor, err_flag: torch.Tensor | None = None,
                   stream=None) -> torch.Tensor:
    """End to end from host tensors (pinned for async copies); sync before reading y_host."""
    B = x_host.shape[0]
    _check("moe_layer_host", lib().moe_layer_host(
        ctypes.byref(weights.shape), ctypes.byref(weights.struct), _ptr(x_host, _BF16, "x_host"),
        _ptr(ids_host, (torch.int32,), "ids_host"), _ptr(wts_host, (torch.float32,), "wts_host"), B,
        _ptr(x_dev, _BF16, "x_dev"), _ptr(ids_dev, (torch.int32,), "ids_dev"),
        _ptr(wts_dev, (torch.float32,), "wts_dev"), _ptr(h_dev, _BF16, "h_dev"),
        _ptr(y_dev, (torch.float32,), "y_dev"), _ptr(y_host, (torch.float32,), "y_host"),
        _ptr(err_flag, (torch.int32,), "err_flag"), _stream(stream)))
    return y_host


def moe_local_ids(shape: MoeShape, ids: torch.Tensor, e_first: int, e_count: int,
                  local_ids: torch.Tensor, err_flag: torch.Tensor | None = None,
                  stream=None) -> torch.Tensor:
    """local_ids[t,j] = ids[t,j] - e_first for the shard's experts, else -1."""
    B = ids.shape[0]
    _check("moe_local_ids", lib().moe_local_ids(
        ctypes.byref(shape), _ptr(ids, (torch.int32,), "ids"), B, e_first, e_count,
        _ptr(local_ids, (torch.int32,), "local_ids"), _ptr(err_flag, (torch.int32,), "err_flag"),
        _stream(stream)))
    return local_ids


def exported_symbols() -> list[str]:
    """The entry points include/warp_decode.h declares."""
    return ["moe_packed_bytes", "moe_pack_weights", "moe_gate_up", "moe_gate_up_grouped",
            "moe_layer_gate_up_kernel", "moe_down", "moe_down_grouped",
            "moe_layer_down_kernel", "moe_layer_host_kernels", "moe_layer",
            "moe_layer_host", "moe_layer_noalloc", "moe_route", "moe_layer_routed",
            "moe_local_ids", "moe_status_string", "moe_last_error"]
