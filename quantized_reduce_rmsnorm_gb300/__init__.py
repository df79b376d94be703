"""libfcomm: quantized tensor-parallel All-Reduce + residual add + RMSNorm on one GB300.

The compute is the C-ABI library libfcomm.so (hand-written sm_103a CUDA,
declared in include/fcomm.h); ``fcomm`` is its thin ctypes binding and
``synth`` draws the seeded synthetic inputs.
"""
from . import build, fcomm, synth  # noqa: F401
from .fcomm import *  # noqa: F401,F403
