"""GB300 (sm_103a) 2-D convolution forward pass behind a cuDNN-style C ABI.

``include/dlc.h`` declares the C ABI; ``binding`` exposes it under the same
names through ctypes; ``api`` builds descriptors from torch tensors; ``synth``
holds the seeded synthetic workloads.  ``build.build()`` compiles the library
into ``_build/libdlc.so``.
"""
__all__ = ["api", "binding", "build", "synth"]
