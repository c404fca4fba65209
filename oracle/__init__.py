"""CPU oracle of the Mamba2 mixer block.  Test infrastructure only: imported by
tests, the package smoke check and the benchmark's CPU-baseline leg, never by
the CUDA library or its Python binding."""
from .m2_oracle import *  # noqa: F401,F403
from . import m2_oracle  # noqa: F401
