"""CPU oracle (test infrastructure): the plain statement of the FP8 linear
path that the CUDA library is checked against.  Imported only by the tests,
the package smoke check and the benchmark's CPU-baseline leg."""
from .fp8_oracle import *  # noqa: F401,F403
