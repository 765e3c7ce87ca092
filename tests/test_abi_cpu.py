"""The C-ABI library without a GPU: symbols, host-side validation, the packer."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from output_centric_expert_gb300 import ops, workload

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "warp_decode.h")


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    declared = _declared_functions()
    assert "moe_gate_up" in declared and "moe_down" in declared and "moe_layer" in declared
    L = ops.lib()
    for name in declared:
        assert hasattr(L, name), f"{name} declared in warp_decode.h but not exported"
    assert sorted(ops.exported_symbols()) == declared


def _fake_weights(aligned=True):
    base = 0x10000 if aligned else 0x10001
    return ops.MoeWeights(base, base + 0x1000, base + 0x2000, base + 0x3000)


def test_host_validation_rejects_before_launch():
    """Bad arguments return an error code and launch nothing (no GPU needed)."""
    L = ops.lib()
    sh = ops.make_shape(256, 128, 8, 2)
    w = _fake_weights()
    P = 0x20000  # 16-byte aligned fake device address (never dereferenced)

    def gate_up(shape, weights, x, ids, B, h, err=None):
        return L.moe_gate_up(ctypes.byref(shape) if shape else None,
                             ctypes.byref(weights) if weights else None, x, ids, B, h, err, None)

    assert gate_up(None, w, P, P, 1, P) == 1  # MOE_ERR_NULL
    assert gate_up(sh, None, P, P, 1, P) == 1
    assert gate_up(sh, w, None, P, 1, P) == 1
    for bad in ((250, 128, 8, 2), (256, 100, 8, 2), (256, 128, 0, 1), (256, 128, 8, 0),
                (8224, 128, 8, 2)):
        assert gate_up(ops.make_shape(*bad), w, P, P, 1, P) == 2  # MOE_ERR_SHAPE
    # top_k may exceed E (ids repeat; an expert-parallel shard holds fewer experts
    # than top_k), but routing from logits needs top_k distinct experts
    assert gate_up(ops.make_shape(256, 128, 8, 9), w, None, None, 0, None) == 0
    assert L.moe_route(ctypes.byref(ops.make_shape(256, 128, 8, 9)), P, 1, P, P, None) == 5
    assert gate_up(sh, w, P, P, -1, P) == 2
    assert gate_up(sh, _fake_weights(aligned=False), P, P, 1, P) == 3  # MOE_ERR_ALIGN
    assert gate_up(sh, w, P + 2, P, 1, P) == 3
    assert gate_up(sh, w, P, P, 1, P + 8) == 3
    assert gate_up(sh, w, P, P + 1, 1, P) == 3
    # empty batch: valid, nothing launched
    assert gate_up(sh, w, None, None, 0, None) == 0
    assert L.moe_down(ctypes.byref(sh), ctypes.byref(w), None, None, None, 0, None, None, None) == 0
    assert L.moe_layer(ctypes.byref(sh), ctypes.byref(w), None, None, None, 0, None, None, None, None) == 0
    assert L.moe_down(ctypes.byref(sh), ctypes.byref(w), P, P, P + 2, 1, P, None, None) == 3
    assert L.moe_layer(ctypes.byref(sh), ctypes.byref(w), P, P, P, 1, None, P, None, None) == 1
    assert "shape" in ops.lib().moe_last_error().decode() or ops.lib().moe_last_error() is not None
    assert ops.status_string(2) == "unsupported shape"


def test_routed_entry_points_validate_before_launch():
    L = ops.lib()
    P = 0x20000
    w = _fake_weights()
    ok = ops.make_shape(2048, 768, 128, 8)
    assert L.moe_route(ctypes.byref(ok), None, 4, P, P, None) == 1          # no logits
    assert L.moe_route(ctypes.byref(ops.make_shape(2048, 768, 512, 8)), P, 4, P, P, None) == 5  # E > 256
    assert L.moe_route(ctypes.byref(ops.make_shape(2048, 768, 128, 40)), P, 4, P, P, None) == 5  # k > 32
    assert L.moe_route(ctypes.byref(ok), P + 2, 4, P, P, None) == 3         # misaligned logits
    assert L.moe_route(ctypes.byref(ok), P, 0, None, None, None) == 0       # empty batch
    assert L.moe_layer_routed(ctypes.byref(ok), ctypes.byref(w), P, P, 4, P, P, P, None, None, None) == 1
    assert L.moe_layer_routed(ctypes.byref(ok), ctypes.byref(w), P, None, 4, P, P, None, None, None, None) == 1


def test_packed_sizes():
    q30 = ops.make_shape(2048, 768, 128, 8)
    sizes = [ops.moe_packed_bytes(q30, w) for w in range(4)]
    assert sizes == [128 * 768 * 2 * 2048, 128 * 768 * 2 * 64, 128 * 2048 * 768, 128 * 2048 * 24]
    per_expert = sum(sizes) // 128
    assert per_expert == 3 * 2048 * 768 + 3 * 2048 * 768 // 32 == 4_866_048
    assert ops.moe_packed_bytes(ops.make_shape(100, 768, 128, 8), 0) == 0
    assert ops.moe_packed_bytes(q30, 7) == 0


def _unpack_to_canonical(packed: ops.PackedHost, H, I, E):
    """Product layout -> the oracle's canonical arrays (layout knowledge only)."""
    gu = packed.gu_codes.reshape(E, I, 2, H)
    gus = packed.gu_scales.reshape(E, I, 2, H // 32)
    return (gu[:, :, 0], gus[:, :, 0], gu[:, :, 1], gus[:, :, 1],
            packed.d_codes.reshape(E, H, I), packed.d_scales.reshape(E, H, I // 32))


@pytest.mark.parametrize("H,I,E", [(256, 128, 8), (64, 96, 3), (32, 32, 1)])
def test_packer_matches_oracle_quantizer_bit_exact(H, I, E):
    rng = np.random.default_rng(H + I + E)
    g = (rng.standard_normal((E, I, H)) * 0.05).astype(np.float32)
    u = (rng.standard_normal((E, I, H)) * 0.05).astype(np.float32)
    d = (rng.standard_normal((E, H, I)) * 0.05).astype(np.float32)
    # edge blocks: zeros, huge, tiny, exact ties of E4M3 (1.0625 is midway 1.0/1.125)
    g[0, 0, :32] = 0.0
    u[0, 0, :32] *= 1e6
    d[0, 0, :32] *= 1e-35
    g[-1, -1, :32] = np.float32(1.0625) * (np.arange(32) % 3 - 1)
    g[-1, -1, 0] = 448.0 / 256.0  # makes the block scale 2^-8 exactly
    sh = ops.make_shape(H, I, E, 1)
    packed = ops.moe_pack_weights(sh, g, u, d)
    gc, gs, uc, us, dc, ds = _unpack_to_canonical(packed, H, I, E)
    ref = oracle.QuantizedLayer.from_fp32(g, u, d)
    for got, want in ((gc, ref.gate_codes), (gs, ref.gate_scales), (uc, ref.up_codes),
                      (us, ref.up_scales), (dc, ref.down_codes), (ds, ref.down_scales)):
        assert np.array_equal(got, want)


def test_packer_per_expert_slices_equal_whole_pack():
    s = workload.SHAPES["tiny"]
    g, u, d = workload.all_weights(s, seed=5)
    sh = ops.make_shape(s.H, s.I, s.E, s.top_k)
    whole = ops.moe_pack_weights(sh, g, u, d)
    parts = ops.empty_packed_host(sh)
    for e in range(s.E):
        ops.moe_pack_weights(sh, g[e:e + 1], u[e:e + 1], d[e:e + 1], out=parts, expert_offset=e)
    for a, b in zip((whole.gu_codes, whole.gu_scales, whole.d_codes, whole.d_scales),
                    (parts.gu_codes, parts.gu_scales, parts.d_codes, parts.d_scales)):
        assert np.array_equal(a, b)


C_CLIENT = r"""
#include <stdio.h>
#include <string.h>
#include "warp_decode.h"

/* every entry point, taken by address: the program links only if all exist */
typedef void (*any_fn)(void);
static const any_fn entry_points[] = {
  (any_fn)moe_packed_bytes, (any_fn)moe_pack_weights, (any_fn)moe_gate_up,
  (any_fn)moe_gate_up_grouped, (any_fn)moe_layer_gate_up_kernel, (any_fn)moe_down,
  (any_fn)moe_down_grouped, (any_fn)moe_layer_down_kernel, (any_fn)moe_layer_host_kernels,
  (any_fn)moe_layer, (any_fn)moe_layer_host, (any_fn)moe_route, (any_fn)moe_layer_routed,
  (any_fn)moe_layer_noalloc, (any_fn)moe_local_ids, (any_fn)moe_status_string,
  (any_fn)moe_last_error,
};

int main(void) {
  moe_shape s = {2048, 768, 128, 8};
  size_t gu = moe_packed_bytes(&s, 0), ds = moe_packed_bytes(&s, 3);
  moe_shape bad = {100, 768, 128, 8};  /* H % 32 != 0 */
  moe_status rc = moe_gate_up(&bad, NULL, NULL, NULL, 1, NULL, NULL, NULL);
  printf("%zu %zu %d %s %d\n", gu, ds, (int)rc, moe_status_string(rc),
         (int)(sizeof entry_points / sizeof entry_points[0]));
  return 0;
}
"""


def test_header_is_plain_c_and_links(tmp_path):
    """The header compiles as C11 (gcc, no C++), a C program links against the
    library with every entry point, and host-only calls behave as documented."""
    import shutil
    import subprocess

    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    lib = ops.lib()._name
    src = tmp_path / "client.c"
    src.write_text(C_CLIENT)
    exe = tmp_path / "client"
    subprocess.run([gcc, "-std=c11", "-Wall", "-Werror", "-pedantic", "-I", os.path.dirname(HEADER),
                    str(src), lib, f"-Wl,-rpath,{os.path.dirname(lib)}", "-o", str(exe)],
                   check=True, capture_output=True, text=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    sh = ops.make_shape(2048, 768, 128, 8)
    assert int(out[0]) == ops.moe_packed_bytes(sh, 0)
    assert int(out[1]) == ops.moe_packed_bytes(sh, 3)
    assert int(out[2]) == 2  # MOE_ERR_SHAPE, before any CUDA call
    assert out[3:5] == ["unsupported", "shape"]
    assert int(out[5]) == len(_declared_functions())


def test_layer_gate_up_kernel_rule():
    """The library's statement of the layer's gate/up kernel (a host-only call):
    the grouped kernel from 8*B*top_k >= 13E (H < 4096) or 2*B*top_k >= 3E
    (H >= 4096) when it takes the shape (H % 256, I % 64), the per-token kernel
    otherwise. The GPU test test_layer_uses_the_grouped_kernel_from_its_switch
    checks that the layer really runs the kernel reported here."""
    q30 = ops.make_shape(2048, 768, 128, 8)
    assert ops.layer_gate_up_kernel(q30, 25) == "per_token"
    assert ops.layer_gate_up_kernel(q30, 26) == "grouped"
    q235 = ops.make_shape(4096, 1536, 128, 8)
    assert ops.layer_gate_up_kernel(q235, 23) == "per_token"
    assert ops.layer_gate_up_kernel(q235, 24) == "grouped"
    assert ops.layer_gate_up_kernel(ops.make_shape(2080, 768, 128, 8), 64) == "per_token"
    assert ops.layer_gate_up_kernel(ops.make_shape(2048, 96, 128, 8), 64) == "per_token"
    assert ops.layer_gate_up_kernel(ops.make_shape(256, 128, 8, 2), 6) == "per_token"
    assert ops.layer_gate_up_kernel(ops.make_shape(256, 128, 8, 2), 7) == "grouped"
    for (H, I, E, k) in [(2048, 768, 128, 8), (4096, 1536, 128, 8), (7168, 2048, 256, 8),
                         (4096, 14336, 8, 2), (256, 128, 8, 2), (768, 192, 5, 3)]:
        sh = ops.make_shape(H, I, E, k)
        for B in (1, 2, 5, 6, 7, 8, 16, 17, 23, 24, 25, 26, 39, 40, 64, 65, 256):
            P = B * k
            shared = (2 * P >= 3 * E) if H >= 4096 else (8 * P >= 13 * E)
            want = "grouped" if (shared and H % 256 == 0 and I % 64 == 0 and E <= 256) else "per_token"
            assert ops.layer_gate_up_kernel(sh, B) == want, (H, I, E, k, B)
    # misaligned scales keep the per-token kernel; a bad shape is an error
    w = ops.MoeWeights(256, 0x1001, 256, 256)
    out = ctypes.c_int32(-1)
    assert ops.lib().moe_layer_gate_up_kernel(ctypes.byref(q30), ctypes.byref(w), 64,
                                              ctypes.byref(out)) == 0 and out.value == 0
    with pytest.raises(ops.WarpDecodeError):
        ops.layer_gate_up_kernel(ops.make_shape(100, 768, 128, 8), 64)


def test_layer_host_kernel_choice():
    """moe_layer_host picks its kernels from the batch's own ids: pairs per used
    expert against the measured break-even points. Uniform routing gives the
    same choice as the rules on B (Qwen-3-30B-A3B shape: per-token up to 24
    tokens, grouped gate/up from 28, both grouped from 40); a skewed batch of 32
    tokens, its pairs on a few dozen experts, takes the grouped kernels; a skewed
    batch of 8 tokens (64 pairs, under 3E/4, and fewer than 4 per used expert)
    keeps the per-token ones; all on one expert takes the grouped ones; no
    valid id keeps the per-token kernels. Host-only."""
    from output_centric_expert_gb300 import workload
    q30 = workload.SHAPES["q30"]
    sh = ops.make_shape(q30.H, q30.I, q30.E, q30.top_k)
    for B in (8, 16, 24):  # 24 tokens: 1.98 pairs per used expert
        ids = workload.tokens(q30, B, seed=0, batch=0, routing="uniform")[1]
        assert ops.layer_host_kernels(sh, ids) == ("per_token", "per_token"), B
    for B in (28, 32, 36):  # 2.13, 2.29 and 2.46 pairs per used expert
        ids = workload.tokens(q30, B, seed=0, batch=0, routing="uniform")[1]
        assert ops.layer_host_kernels(sh, ids) == ("grouped", "per_token"), B
        assert ops.layer_gate_up_kernel(sh, B) == "grouped" and ops.layer_down_kernel(sh, B) == "per_token"
    for B in (40, 48, 64):
        ids = workload.tokens(q30, B, seed=0, batch=0, routing="uniform")[1]
        assert ops.layer_host_kernels(sh, ids) == ("grouped", "grouped"), B
        assert ops.layer_gate_up_kernel(sh, B) == "grouped" and ops.layer_down_kernel(sh, B) == "grouped"
    for b in range(4):
        ids = workload.tokens(q30, 32, seed=0, batch=b, routing="skewed")[1]
        U = len(np.unique(ids))
        assert 256 >= 2.6 * U, U  # the skewed batches crowd onto few experts
        assert ops.layer_host_kernels(sh, ids) == ("grouped", "grouped")
        ids = workload.tokens(q30, 8, seed=0, batch=b, routing="skewed")[1]
        assert 2.0 * len(np.unique(ids)) <= 64 < 4 * len(np.unique(ids))  # 2.0-2.4 per used expert
        assert ops.layer_host_kernels(sh, ids) == ("per_token", "per_token")
    one = np.full((8, 8), 5, dtype=np.int32)  # 64 pairs on expert 5 (duplicates within tokens)
    assert ops.layer_host_kernels(sh, one) == ("grouped", "grouped")
    none = np.full((8, 8), -1, dtype=np.int32)
    assert ops.layer_host_kernels(sh, none) == ("per_token", "per_token")
    # the thresholds in pairs per used expert, at a boundary (top_k = 1, 8 experts,
    # so that 3E/4 = 6 pairs): down grouped from 2.6 per expert (13 pairs on 5
    # experts; 12 on 5 is 2.4), gate/up from 2.0 (10 on 5; 9 on 5 is 1.8)
    sh1 = ops.make_shape(2048, 768, 8, 1)
    ids13 = np.array([[e] for e in [0, 1, 2, 3, 4] * 2 + [0, 1, 2]], dtype=np.int32)
    assert ops.layer_host_kernels(sh1, ids13) == ("grouped", "grouped")
    assert ops.layer_host_kernels(sh1, ids13[:12]) == ("grouped", "per_token")
    assert ops.layer_host_kernels(sh1, ids13[:10]) == ("grouped", "per_token")
    assert ops.layer_host_kernels(sh1, ids13[:9]) == ("per_token", "per_token")
    # below 3E/4 pairs only 4 pairs per used expert or more count: 13 pairs on 5
    # of 128 experts keep the per-token kernels, 20 on 5 take the grouped ones
    sh1b = ops.make_shape(2048, 768, 128, 1)
    assert ops.layer_host_kernels(sh1b, ids13) == ("per_token", "per_token")
    ids20 = np.array([[e] for e in [0, 1, 2, 3, 4] * 4], dtype=np.int32)
    assert ops.layer_host_kernels(sh1b, ids20) == ("grouped", "grouped")
    # longer rows: gate/up from 1.95 pairs per expert (H >= 4096), down from 2.2 (H >= 6144)
    sh4 = ops.make_shape(4096, 1536, 8, 1)
    ids9 = np.array([[e] for e in [0, 1, 2, 3] * 2 + [0]], dtype=np.int32)  # 9 on 4: 2.25
    assert ops.layer_host_kernels(sh4, ids9) == ("grouped", "per_token")
    sh4b = ops.make_shape(4096, 1536, 32, 1)
    ids39 = np.array([[e] for e in list(range(20)) + list(range(19))], dtype=np.int32)  # 39 on 20
    assert ops.layer_host_kernels(sh4b, ids39)[0] == "grouped"  # 1.95 pairs per used expert
    assert ops.layer_host_kernels(sh4b, ids39[:38])[0] == "per_token"  # 1.9
    sh7 = ops.make_shape(7168, 2048, 8, 1)
    assert ops.layer_host_kernels(sh7, ids9) == ("grouped", "grouped")
    assert ops.layer_host_kernels(sh7, ids9[:8]) == ("grouped", "per_token")  # 2.0 per expert
    # intermediate rows of 3H and more: down from 1.5 pairs per expert
    shm = ops.make_shape(4096, 14336, 8, 1)
    ids6 = np.array([[e] for e in [0, 1, 2, 3, 0, 1]], dtype=np.int32)  # 6 on 4
    assert ops.layer_host_kernels(shm, ids6) == ("per_token", "grouped")
    assert ops.layer_host_kernels(shm, ids6[:5]) == ("per_token", "per_token")  # 5 < 3E/4
    # E > 256: beyond the grouped kernels
    big = ops.make_shape(2048, 768, 257, 8)
    assert ops.layer_host_kernels(big, one) == ("per_token", "per_token")
    with pytest.raises(ops.WarpDecodeError):
        ops.layer_host_kernels(ops.make_shape(100, 768, 128, 8), one)


def test_layer_host_kernel_rule_on_random_batches():
    """moe_layer_host_kernels follows the rule the header states, on random
    batches of up to 64 tokens whose ids crowd onto random subsets of the
    experts (some slots invalid): with P = B*top_k pairs and U distinct valid
    experts, either step is grouped only when 4P >= 3E or P >= 4U, gate/up
    when P >= 2U (H < 4096) or 20P >= 39U (H >= 4096), down when 2P >= 3U
    (I >= 3H), else 5P >= 13U (H < 6144) or 5P >= 11U (H >= 6144). The shapes
    are ones both grouped kernels take at 64 tokens (checked). Host-only."""
    rng = np.random.default_rng(7)
    shapes = [(2048, 768, 128, 8), (4096, 1536, 128, 8), (7168, 2048, 256, 8),
              (4096, 14336, 8, 2), (2048, 768, 16, 4), (7168, 2048, 64, 2)]
    for (H, I, E, k) in shapes:
        sh = ops.make_shape(H, I, E, k)
        assert ops.layer_gate_up_kernel(sh, 64) == "grouped" and ops.layer_down_kernel(sh, 64) == "grouped"
        for _ in range(60):
            B = int(rng.integers(1, 65))
            pool = rng.choice(E, size=int(rng.integers(1, E + 1)), replace=False)
            ids = rng.choice(pool, size=(B, k)).astype(np.int32)
            ids[rng.random((B, k)) < 0.05] = -1
            P = B * k
            U = len(np.unique(ids[ids >= 0]))
            enough = U > 0 and (4 * P >= 3 * E or P >= 4 * U)
            gu = enough and ((20 * P >= 39 * U) if H >= 4096 else (P >= 2 * U))
            dn = enough and ((2 * P >= 3 * U) if I >= 3 * H else
                             (5 * P >= 11 * U) if H >= 6144 else (5 * P >= 13 * U))
            want = ("grouped" if gu else "per_token", "grouped" if dn else "per_token")
            assert ops.layer_host_kernels(sh, ids) == want, (H, I, E, k, B, U)


def test_layer_down_kernel_choice():
    """The layer's down kernel: the expert-grouped one from 2.5E pairs (2E for
    rows of 6144 and more; 1.25E where the intermediate rows are 3H or longer)
    when it takes the shape (I % 256 == 0, E <= 256) and batch (up to 64 tokens for
    these shapes; never beyond 128), the per-token one otherwise; the library
    answers on the host, without a GPU."""
    for (H, I, E, k) in [(2048, 768, 128, 8), (4096, 1536, 128, 8), (7168, 2048, 256, 8),
                         (4096, 14336, 8, 2), (256, 128, 8, 2), (64, 256, 6, 3),
                         (2048, 768, 257, 8)]:
        sh = ops.make_shape(H, I, E, k)
        for B in (1, 2, 3, 4, 5, 9, 10, 15, 16, 17, 32, 39, 40, 63, 64, 129, 256):
            P = B * k
            shared = (4 * P >= 5 * E) if I >= 3 * H else \
                (P >= 2 * E) if H >= 6144 else (2 * P >= 5 * E)
            want = "grouped" if (shared and I % 256 == 0 and E <= 256 and B <= 64) \
                else "per_token"
            assert ops.layer_down_kernel(sh, B) == want, (H, I, E, k, B)
    # misaligned down scales keep the per-token kernel; NULL weight arrays and
    # a bad shape are errors
    q30 = ops.make_shape(2048, 768, 128, 8)
    out = ctypes.c_int32(-1)
    w = ops.MoeWeights(256, 256, 256, 0x1001)
    assert ops.lib().moe_layer_down_kernel(ctypes.byref(q30), ctypes.byref(w), 64,
                                           ctypes.byref(out)) == 0 and out.value == 0
    w = ops.MoeWeights(256, 256, 256, None)
    assert ops.lib().moe_layer_down_kernel(ctypes.byref(q30), ctypes.byref(w), 64,
                                           ctypes.byref(out)) == 1
    w = ops.MoeWeights(256, None, 256, 256)
    assert ops.lib().moe_layer_gate_up_kernel(ctypes.byref(q30), ctypes.byref(w), 64,
                                              ctypes.byref(out)) == 1
    with pytest.raises(ops.WarpDecodeError):
        ops.layer_down_kernel(ops.make_shape(100, 768, 128, 8), 64)
