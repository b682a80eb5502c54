"""libswa: sliding-window (BAND) / unmasked FlashAttention forward and backward
for GB300 (sm_103a), hand-written CUDA behind a C ABI (include/swa.h).

``swa`` is the ctypes binding (the compiled library loads on first use);
``workloads`` draws seeded synthetic inputs; ``build`` compiles libswa.so.
"""
from . import swa  # noqa: F401
from .swa import SwaError, backward, forward  # noqa: F401
