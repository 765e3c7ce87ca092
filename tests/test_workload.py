"""The seeded input generator: published splitmix64 outputs, determinism, laws."""
import numpy as np

from output_centric_expert_gb300 import workload


def test_splitmix64_published_sequence():
    # First outputs of splitmix64 from state 0 (Vigna's reference splitmix64.c)
    expect = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F, 0xF88BB8A8724C81EC]
    assert [workload.splitmix64_at(0, i) for i in range(4)] == expect


def test_normals_are_standard():
    key = workload.stream_key(0, 99)
    z = workload.normal_f32(key, 0, 200_000).astype(np.float64)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1) < 0.01
    # counter-based: a window equals the same slice of a longer draw
    np.testing.assert_array_equal(workload.normal_f32(key, 1000, 50), z[1000:1050].astype(np.float32))


def test_expert_weights_independent_of_generation_order():
    s = workload.SHAPES["tiny"]
    g, u, d = workload.all_weights(s, seed=3)
    g5, u5, d5 = workload.expert_weights(s, 5, seed=3)
    np.testing.assert_array_equal(g[5], g5)
    np.testing.assert_array_equal(u[5], u5)
    np.testing.assert_array_equal(d[5], d5)
    assert g.shape == (8, 128, 256) and d.shape == (8, 256, 128)
    assert not np.array_equal(g, u)
    assert abs(float(g.std()) - workload.WEIGHT_STD) < 2e-3
    # another layer index gives other weights
    g2, _, _ = workload.expert_weights(s, 5, seed=3, layer=1)
    assert not np.array_equal(g2, g5)


def test_routing_laws():
    s = workload.SHAPES["q30"]
    for routing in ("uniform", "skewed"):
        x, ids, w = workload.tokens(s, 64, seed=0, routing=routing)
        assert x.shape == (64, 2048) and x.dtype == np.uint16
        assert ids.shape == (64, 8) and ids.dtype == np.int32
        assert np.all((ids >= 0) & (ids < s.E))
        assert all(len(set(r)) == s.top_k for r in ids.tolist())
        np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=1e-6)
        assert np.all(np.diff(w, axis=1) <= 0)  # descending routing probability
    _, ids_u, _ = workload.tokens(s, 64, routing="uniform")
    _, ids_s, _ = workload.tokens(s, 64, routing="skewed")
    assert len(np.unique(ids_s)) < len(np.unique(ids_u))  # hot experts shared
    # deterministic, and batches differ
    a = workload.tokens(s, 4, seed=0, batch=0)
    b = workload.tokens(s, 4, seed=0, batch=0)
    c = workload.tokens(s, 4, seed=0, batch=1)
    assert all(np.array_equal(p, q) for p, q in zip(a, b))
    assert not np.array_equal(a[0], c[0])


def test_empty_batch_tokens():
    x, ids, w = workload.tokens(workload.SHAPES["tiny"], 0)
    assert x.shape == (0, 256) and ids.shape == (0, 2) and w.shape == (0, 2)
