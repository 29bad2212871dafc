"""RidgeFill upper-layer KV fill, calibration, ridge solve and cross-model mapper on
GB300 (sm_103a). The compute path is librf.so (include/rf.h); this package is its
ctypes binding plus the build step. There is no CPU fallback."""
from ._binding import *  # noqa: F401,F403
from ._binding import LIB_PATH, RFError, lib  # noqa: F401

__version__ = "0.1.0"
