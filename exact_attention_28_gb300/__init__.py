"""FlashAttention forward for one NVIDIA GB300 (sm_103a).

The compute path is the C-ABI library ``libfa_gb300.so`` built from ``csrc/``
(hand-written CUDA: TMA loads, tcgen05 MMAs accumulating in tensor memory,
online softmax).  ``ops`` is a thin ctypes binding with the same names as the
C entry points; it only marshals arguments.  There is no CPU fallback: if the
library is missing, every call raises.
"""
from __future__ import annotations

__all__ = ["ops", "inputs"]


def __getattr__(name):
    if name in ("ops", "inputs"):
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
