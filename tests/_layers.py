"""Test helper: one seeded layer, packed twice from the same FP32 weights.

* the product packer writes the device layout the CUDA path reads;
* the oracle's own quantiser writes the canonical arrays the oracle reads.

The two never exchange data (they agree bit for bit, which the CPU tests
check separately). Only the experts the oracle will need are quantised for it.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

import oracle
from output_centric_expert_gb300 import ops, workload


class Layer:
    def __init__(self, shape: workload.LayerShape, seed: int = 0, layer: int = 0,
                 oracle_experts=None, device: str = "cuda"):
        self.shape = shape
        self.sh = ops.make_shape(shape.H, shape.I, shape.E, shape.top_k)
        E, I, H = shape.E, shape.I, shape.H
        packed = ops.empty_packed_host(self.sh)
        need = set(range(E)) if oracle_experts is None else set(int(e) for e in oracle_experts)
        gc = np.zeros((E, I, H), np.uint8)
        gs = np.zeros((E, I, H // 32), np.uint8)
        uc, us = np.zeros_like(gc), np.zeros_like(gs)
        dc = np.zeros((E, H, I), np.uint8)
        ds = np.zeros((E, H, I // 32), np.uint8)

        def one(e):
            g, u, d = workload.expert_weights(shape, e, seed, layer)
            ops.moe_pack_weights(self.sh, g[None], u[None], d[None], out=packed, expert_offset=e)
            if e in need:
                gc[e], gs[e] = oracle.quantize_mxfp8(g)
                uc[e], us[e] = oracle.quantize_mxfp8(u)
                dc[e], ds[e] = oracle.quantize_mxfp8(d)

        with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
            list(ex.map(one, range(E)))
        self.packed = packed
        self.ref = oracle.QuantizedLayer(gc, gs, uc, us, dc, ds)
        self.dev = ops.DeviceWeights(self.sh, packed, device) if device else None


def parity_stats(y_gpu: np.ndarray, y_ref: np.ndarray):
    """max |y_gpu - y_ref| and the minimum per-token cosine similarity."""
    y_gpu = y_gpu.astype(np.float64)
    d = float(np.max(np.abs(y_gpu - y_ref))) if y_ref.size else 0.0
    num = np.sum(y_gpu * y_ref, axis=1)
    den = np.linalg.norm(y_gpu, axis=1) * np.linalg.norm(y_ref, axis=1)
    cos = np.where(den > 0, num / np.where(den > 0, den, 1), 1.0)
    return d, float(cos.min()) if cos.size else 1.0
