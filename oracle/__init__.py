"""fp64 C++ CPU oracle (test infrastructure only; see llama_oracle.h for its sources and readings)."""
from .llama_oracle import *  # noqa: F401,F403
from .llama_oracle import Dims, BlockWeights, block_rows, threads  # noqa: F401
from . import sampling  # noqa: F401
from . import fp8  # noqa: F401
from ._lib import build  # noqa: F401
