"""CPU oracle of the quantized attention contract (test infrastructure only)."""
from .sage_oracle import *  # noqa: F401,F403
