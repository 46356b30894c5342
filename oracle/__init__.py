"""CPU fp64 oracle (test infrastructure only; never on the product path)."""
from .ttt_oracle import *  # noqa: F401,F403
