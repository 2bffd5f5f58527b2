"""fp64 CPU oracle (test infrastructure only; see quest_oracle's docstring)."""

from .quest_oracle import *  # noqa: F401,F403
from . import quest_oracle  # noqa: F401
