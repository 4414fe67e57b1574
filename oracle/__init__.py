"""fp64 CPU oracle (test infrastructure only; see sv_oracle.py)."""
from .sv_oracle import *  # noqa: F401,F403
