"""fp64 CPU oracle (test infrastructure only; see llama_oracle.py's header)."""
from .llama_oracle import *  # noqa: F401,F403
from .llama_oracle import Dims, BlockWeights  # noqa: F401
from . import sampling  # noqa: F401
from . import fp8  # noqa: F401
