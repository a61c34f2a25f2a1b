"""CPU oracle (test infrastructure only; see zero_oracle.py's header)."""
from .zero_oracle import *  # noqa: F401,F403
