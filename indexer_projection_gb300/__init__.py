"""GB300 (sm_103a) MiniMax-M3 sparse-layer pre-attention step.

The compute lives in libpre_attn.so (hand-written CUDA, C-ABI in
include/pre_attn.h); ``binding`` is its ctypes mirror and ``runner`` a thin
torch-tensor front end (device memory and streams only).
"""

from . import binding  # noqa: F401

__all__ = ["binding", "runner", "build"]
