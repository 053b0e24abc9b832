"""CPU oracle of the MoE-layer hot path (test infrastructure only).

Importable by the tests, the package's smoke check and the benchmark's CPU
baseline; never by the library itself.
"""
from .moe_oracle import *  # noqa: F401,F403
