"""fp64 CPU oracle (test infrastructure only; see rowpass_oracle's header)."""
from .rowpass_oracle import *  # noqa: F401,F403
