"""fp64 CPU oracle of the low-rank bottleneck sublayer.

TEST INFRASTRUCTURE ONLY: tests, the smoke check and the benchmark's CPU
baseline leg use it; the CUDA library never does.
"""
from .lowrank_oracle import *  # noqa: F401,F403
from .lowrank_oracle import mlp_block_rows  # noqa: F401
