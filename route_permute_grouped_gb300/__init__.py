"""GB300-native MoE layer hot path: route -> permute -> grouped SwiGLU experts ->
combine, and the training backward, as hand-written sm_103a CUDA behind a C ABI.

Importing the package loads nothing; ``route_permute_grouped_gb300.ops`` binds the
compiled library and raises if it is missing.
"""
__all__ = ["synth", "ops", "build"]
