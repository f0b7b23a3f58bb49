"""CPU float64 oracle (test infrastructure only; see txl_oracle)."""
from .txl_oracle import *  # noqa: F401,F403
