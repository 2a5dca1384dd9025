"""CPU oracle (test infrastructure only; see mxfp8_oracle.py). The CUDA library never
imports this package."""
from .mxfp8_oracle import *  # noqa: F401,F403
