"""CPU fp64 oracle (test infrastructure only; see kvc_oracle's header)."""
from .kvc_oracle import *  # noqa: F401,F403
