"""DeepSeekMoE layer forward on one B300 (sm_103a).

The compute path lives in ``libmoe.so`` (hand-written CUDA behind a C ABI,
``include/moe.h``).  ``ops`` is a thin ctypes binding with the same entry
point names; importing this package does not load the library, the first op
call does, and it raises if the library is missing -- there is no fallback.
"""
__all__ = ["inputs", "ops"]
