"""CPU oracle (test infrastructure only; see fp8q_oracle.py's header)."""
from .fp8q_oracle import *  # noqa: F401,F403
from . import fp8q_oracle  # noqa: F401
