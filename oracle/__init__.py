"""fp64 CPU oracle of the fused MoE expert layer (forward, backward, MXFP8 quantise-dequantise).

TEST INFRASTRUCTURE ONLY. It exists to check the CUDA path, never to stand in for it: only the
tests, the smoke check and the CPU-baseline / reference legs of the benchmark may import it.
It shares no code, table or helper with the CUDA library and imports nothing from it.
"""
from .moe_oracle import *  # noqa: F401,F403
