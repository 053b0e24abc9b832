"""GB300-native (sm_103a) MoE-layer hot path.

router GEMM -> top-K routing -> permute -> grouped SwiGLU expert GEMM ->
weighted unpermute/combine, as hand-written CUDA kernels behind a C ABI
(``include/moe_gb300.h``).  ``ops`` is the thin ctypes binding; ``synth`` draws
seeded synthetic inputs.
"""
__all__ = ["ops", "synth", "build"]
