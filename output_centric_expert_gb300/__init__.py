"""GB300-native output-centric ("warp decode") MoE decode layer.

The layer is two hand-written CUDA kernels for sm_103a behind a C ABI
(``include/warp_decode.h``, built into ``_build/libwarp_decode.so``):

* ``moe_gate_up`` -- one warp per (token, routed expert, intermediate neuron):
  gate and up dot products from one read of the BF16 activation against MXFP8
  weights decoded on the fly, SiLU(gate)*up written as BF16;
* ``moe_down`` -- one warp per (token, output dim): one FP32 accumulator streamed
  over all top-k experts' down rows with the routing weight folded in, finished
  by a warp butterfly. No padding, gather, scatter or combine buffers exist.

``ops`` is the thin Python binding (argument marshalling only); ``workload``
is the seeded synthetic input generator. Importing this package loads nothing
native: the CUDA library is built/loaded on first use and any failure raises.
"""

__all__ = ["ops", "workload"]


def __getattr__(name):
    if name in ("ops", "workload"):
        import importlib

        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
