"""Expert parallelism for the MoE decode layer: the layer split over G devices.

Each device holds a contiguous range of the E experts (the packed MXFP8
layout is expert-major, so a shard is a slice of each packed array). For a
batch, every device computes the slots routed to its own experts: the
C-ABI call ``moe_local_ids`` maps the global expert ids to the shard's local
ids (-1 for a slot on another device, which the layer kernels skip as they
skip an invalid id), the layer runs on the shard with no error flag (the
mapping flags ids outside [0, E)), and one all-reduce (sum) of y [B, H] FP32
across the devices gives the layer's output. The combine is exact up to FP32
rounding order because the layer is linear in its slots.

The pages describe no multi-device split ("Better MoE model inference with
warp decode" measures one B200); this is the split the expert-major layout
allows with a single exchange. This module holds host logic only: the device
work is the library's kernels and torch.distributed's all-reduce.
"""
from __future__ import annotations

from typing import Callable

import numpy as np


def shard_range(E: int, rank: int, world: int) -> tuple[int, int]:
    """(e_first, e_count): the contiguous experts of device `rank` of `world`;
    the first E % world devices hold one expert more."""
    if not (0 <= rank < world) or world > E:
        raise ValueError(f"need 0 <= rank < world <= E (rank {rank}, world {world}, E {E})")
    base, extra = divmod(E, world)
    e_first = rank * base + min(rank, extra)
    return e_first, base + (1 if rank < extra else 0)


def shard_packed(packed, shape, e_first: int, e_count: int):
    """The packed arrays of experts [e_first, e_first + e_count) (views into
    `packed`, an ops.PackedHost of all E experts)."""
    from . import ops

    per = [ops.moe_packed_bytes(ops.make_shape(shape.H, shape.I, 1, 1), w) for w in range(4)]
    arrs = (packed.gu_codes, packed.gu_scales, packed.d_codes, packed.d_scales)
    return ops.PackedHost(*(a[e_first * n:(e_first + e_count) * n] for a, n in zip(arrs, per)))


def ep_layer(local_weights, x, ids, wts, h, y, e_first: int, e_count: int, *, global_E: int,
             local_ids=None, err_flag=None, group=None,
             layer: Callable | None = None, remap: Callable | None = None, all_reduce=True):
    """One device's part of the expert-parallel layer, then the all-reduce of y.

    local_weights: this device's experts (E = e_count); ids [B, top_k] global.
    layer(local_weights, x, local_ids, wts, h, y) and remap(global_shape, ids,
    e_first, e_count, local_ids, err_flag) default to the library's moe_layer
    and moe_local_ids; tests may pass other implementations of the same
    contract. Returns y (summed over the process group when all_reduce)."""
    from . import ops

    if layer is None:
        layer = lambda w, x_, i, wt, h_, y_: ops.moe_layer(w, x_, i, wt, h_, y_)  # noqa: E731
    if remap is None:
        remap = ops.moe_local_ids
    gshape = ops.make_shape(local_weights.shape.H, local_weights.shape.I, global_E,
                            local_weights.shape.top_k)
    if local_ids is None:
        local_ids = ids.new_empty(ids.shape) if hasattr(ids, "new_empty") else np.empty_like(ids)
    remap(gshape, ids, e_first, e_count, local_ids, err_flag)
    layer(local_weights, x, local_ids, wts, h, y)
    if all_reduce:
        import torch.distributed as dist

        dist.all_reduce(y, op=dist.ReduceOp.SUM, group=group)
    return y
