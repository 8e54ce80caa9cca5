"""fp64 CPU oracle (test infrastructure only; see coda_oracle's header)."""
from .coda_oracle import *  # noqa: F401,F403
