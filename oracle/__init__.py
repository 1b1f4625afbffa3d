"""fp64 CPU oracle of the MoE FFN layer -- test infrastructure only.

Only the tests, the smoke check and the benchmark's CPU-baseline / reference
arm may import this package.  The CUDA library and its binding never do.
"""

from .moe_oracle import *  # noqa: F401,F403
from .moe_oracle import __all__  # noqa: F401
