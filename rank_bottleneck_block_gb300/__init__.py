"""GB300-native low-rank bottleneck sublayer (BOOST hot path).

The compute path lives in ``liblowrank.so`` (hand-written sm_103a kernels behind
a C ABI, declared in ``include/lowrank.h``).  ``lowrank`` is the thin ctypes
binding; ``inputs`` draws seeded synthetic tensors.  Submodules are imported
lazily so that ``inputs`` can be used without loading the CUDA library.
"""
__all__ = ["inputs", "lowrank", "build"]
