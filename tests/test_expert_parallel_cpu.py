"""Expert parallelism on CPU: the shard arithmetic, and the whole split-and-sum
path on two gloo ranks with the oracle as each rank's layer.

Each rank holds a contiguous range of the experts, computes only the slots
routed to them (the others mapped to -1, which contribute nothing), and one
all-reduce of y gives the layer. The sum must equal the oracle's layer over
all experts.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from output_centric_expert_gb300 import expert_parallel as ep
from output_centric_expert_gb300 import ops, workload


@pytest.mark.parametrize("E,world", [(8, 2), (128, 8), (5, 3), (7, 7), (256, 32)])
def test_shard_ranges_cover_the_experts_once(E, world):
    seen = []
    for r in range(world):
        first, count = ep.shard_range(E, r, world)
        assert count >= 1
        seen += list(range(first, first + count))
    assert seen == list(range(E))


def test_shard_range_rejects_more_devices_than_experts():
    with pytest.raises(ValueError):
        ep.shard_range(4, 0, 5)


def test_shard_of_the_packed_weights_equals_packing_the_shard_alone():
    s = workload.LayerShape(64, 64, 5, 2)
    sh = ops.make_shape(s.H, s.I, s.E, s.top_k)
    g, u, d = workload.all_weights(s, seed=4)
    full = ops.moe_pack_weights(sh, g, u, d)
    for r in range(2):
        first, count = ep.shard_range(s.E, r, 2)
        part = ep.shard_packed(full, s, first, count)
        alone = ops.moe_pack_weights(ops.make_shape(s.H, s.I, count, s.top_k),
                                     g[first:first + count], u[first:first + count],
                                     d[first:first + count])
        for a, b in zip((part.gu_codes, part.gu_scales, part.d_codes, part.d_scales),
                        (alone.gu_codes, alone.gu_scales, alone.d_codes, alone.d_scales)):
            assert np.array_equal(a, b)


def _free_port():
    with socket.socket() as so:
        so.bind(("127.0.0.1", 0))
        return so.getsockname()[1]


def _remap_reference(gshape, ids, e_first, e_count, local_ids, err_flag):
    """The mapping moe_local_ids defines, written out for the CPU ranks."""
    inside = (ids >= e_first) & (ids < e_first + e_count)
    local_ids[...] = np.where(inside, ids - e_first, -1)


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        s = workload.LayerShape(64, 64, 5, 2)
        g, u, d = workload.all_weights(s, seed=4)
        full = oracle.QuantizedLayer.from_fp32(g, u, d)
        x, ids, w = workload.tokens(s, 6, seed=9)
        ids = ids.copy()
        ids[2, 1] = ids[2, 0]  # a duplicate id
        first, count = ep.shard_range(s.E, rank, world)
        shard = oracle.QuantizedLayer(
            full.gate_codes[first:first + count], full.gate_scales[first:first + count],
            full.up_codes[first:first + count], full.up_scales[first:first + count],
            full.down_codes[first:first + count], full.down_scales[first:first + count])
        shard.shape = ops.make_shape(s.H, s.I, count, s.top_k)

        def layer(wts_, x_, local_ids, w_, h_, y_):
            y_np, _ = oracle.moe_layer(wts_, x_, local_ids, w_)
            y_.copy_(torch.from_numpy(y_np))

        y = torch.zeros((6, s.H), dtype=torch.float64)
        local = np.empty_like(ids)
        ep.ep_layer(shard, x, ids, w, None, y, first, count, global_E=s.E, local_ids=local,
                    layer=layer, remap=_remap_reference)
        y_full, _ = oracle.moe_layer(full, x, ids, w)
        out[rank] = (float(np.max(np.abs(y.numpy() - y_full))), float(np.max(np.abs(y_full))),
                     int((local >= 0).sum()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_split_the_experts_and_the_sum_is_the_layer():
    world = 2
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        diff, scale, _ = res[r]
        assert diff <= 1e-12 * scale, res
    # every slot is local to exactly one rank
    assert res[0][2] + res[1][2] == 6 * 2
