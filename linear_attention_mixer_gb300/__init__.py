"""KDA (Kimi Delta Attention) mixer core for GB300 (sm_103a).

The compute lives in libkda.so (hand-written CUDA behind the C ABI of
include/kda.h); this package holds its sources (csrc/), the nvcc build
(build.py) and the ctypes binding (kda.py).
"""
from .kda import *  # noqa: F401,F403
from .kda import KdaError, lib  # noqa: F401
