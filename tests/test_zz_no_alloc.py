"""The allocation-free layer entry point, moe_layer_noalloc.

Some callers cannot allocate device memory: code running inside a host
framework that owns every device allocation through its own pool, or a
latency-critical decode loop that must not call cudaMalloc. For them the
library keeps the layer's intermediate in a fixed array of its own. These
tests call that entry point through the C ABI and check it against
moe_layer (which takes a caller-provided intermediate buffer) bit for bit on
several calls in a row, so that a call cannot silently reuse an earlier
call's data, and against the CPU oracle on sampled tokens.

This file is collected last on purpose: it runs after every other test.
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


@pytest.fixture(scope="module")
def q30():
    return Layer(workload.SHAPES["q30"])


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("routing", ["uniform", "skewed"])
def test_noalloc_matches_moe_layer_on_two_calls_in_a_row(q30, routing):
    """Three calls in a row (64, 32 and 5 tokens): each must equal moe_layer on
    the same inputs bit for bit (the same kernels run; at 64 tokens the
    expert-grouped kernels write into the library's own array), so a call
    that reused the previous call's intermediate would show. Sampled tokens
    are also checked against the oracle."""
    s = q30.shape
    for B, batch in ((64, 100), (32, 101), (5, 102)):
        x, ids, w = workload.tokens(s, B, batch=batch, routing=routing)
        xd, idd, wd = _dev(x.view(np.int16)), _dev(ids), _dev(w)
        h = torch.empty((B, s.top_k, s.I), dtype=torch.int16, device="cuda")
        y_ref = torch.empty((B, s.H), dtype=torch.float32, device="cuda")
        ops.moe_layer(q30.dev, xd, idd, wd, h, y_ref)
        y = torch.full((B, s.H), float("nan"), dtype=torch.float32, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        ops.moe_layer_noalloc(q30.dev, xd, idd, wd, y, err)
        torch.cuda.synchronize()
        assert np.array_equal(y.cpu().numpy(), y_ref.cpu().numpy()), (B, routing)
        assert int(err.item()) == 0
        sample = sorted({0, B // 2, B - 1})
        y_or, _ = oracle.moe_layer(q30.ref, x[sample], ids[sample], w[sample])
        d, cos = parity_stats(y.cpu().numpy()[sample], y_or)
        assert d <= MAX_ABS and cos >= MIN_COS, (B, routing, d, cos)


def test_noalloc_rejects_an_intermediate_beyond_its_capacity(q30):
    s = q30.shape
    B = ops.MOE_NOALLOC_MAX_INTERMEDIATE // (s.top_k * s.I) + 1  # one token too many
    x = torch.zeros((B, s.H), dtype=torch.int16, device="cuda")
    ids = torch.zeros((B, s.top_k), dtype=torch.int32, device="cuda")
    w = torch.zeros((B, s.top_k), dtype=torch.float32, device="cuda")
    y = torch.zeros((B, s.H), dtype=torch.float32, device="cuda")
    with pytest.raises(ops.WarpDecodeError) as ei:
        ops.moe_layer_noalloc(q30.dev, x, ids, w, y)
    assert ei.value.status == 2 and "capacity" in str(ei.value)
