"""CPU oracle (test infrastructure only; see clover_oracle.py)."""
from .clover_oracle import *  # noqa: F401,F403
