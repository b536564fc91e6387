"""CPU oracle for the sparse MoE FFN layer: test infrastructure only.

Only the test suite, the package smoke check and the benchmark's CPU-baseline
and reference legs may import this package. See ``moe_oracle`` for the
definitions and the readings taken where the source pages are silent.
"""
from .moe_oracle import *  # noqa: F401,F403
from . import moe_oracle  # noqa: F401
