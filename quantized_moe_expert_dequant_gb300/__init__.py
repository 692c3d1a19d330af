"""GB300 (sm_103a) decode MoE expert block over packed affine-quantized experts.

``synth`` and ``workloads`` are plain Python; everything that computes lives in the CUDA library
``libmoe_decode.so`` behind the C ABI in ``include/moe_decode.h``, reached through ``binding``.
Importing the package loads nothing; the binding loads the library on first use and raises if
it is missing.
"""
__all__ = ["synth", "workloads", "binding"]
