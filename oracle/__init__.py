"""fp64 CPU oracle (test infrastructure only; never part of the product path)."""
from .oracle import *  # noqa: F401,F403
