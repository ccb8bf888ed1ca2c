"""CPU oracle for AWQ's per-layer scale search and INT4 packing.

TEST INFRASTRUCTURE ONLY: imported by the tests, the package smoke check and
the benchmark's CPU-baseline leg, never by the library's compute path.
"""
from .awq_oracle import *  # noqa: F401,F403
from .awq_oracle import __all__  # noqa: F401
