"""CPU oracle for the Q4_K x Q8_1 decode path -- TEST INFRASTRUCTURE ONLY.

Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
import this package.  The product path (the CUDA library and its binding) never
does, and shares no code with it.

Each function marshals numpy arrays into the plain C oracle in rz_oracle.c
(single-threaded, double accumulation, f32 at the step boundaries where the
method passes f32 buffers).  See rz_oracle.c for the passages each step follows.
"""
from .api import *  # noqa: F401,F403
from .api import __all__  # noqa: F401
