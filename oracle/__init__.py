"""fp64 CPU oracle (test infrastructure only; see ridgefill.py)."""
from .ridgefill import *  # noqa: F401,F403
from .ridgefill import add_stats  # noqa: F401
