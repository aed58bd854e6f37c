"""fp64 CPU oracle for the MoE layer hot path (route, permute, grouped SwiGLU
experts, combine, and the training backward).

TEST INFRASTRUCTURE. This package is the independent checker of the CUDA path.
Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
import it. It shares no code with the CUDA library and imports nothing from it.

Method source: "Scalable Training of Mixture-of-Experts Models with Megatron
Core" (paper summary page and the figures & tables page of the same report).
"""
from .moe_oracle import *  # noqa: F401,F403
from .mx_oracle import *  # noqa: F401,F403
from .nv_oracle import *  # noqa: F401,F403
