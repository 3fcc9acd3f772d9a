"""Exact greedy speculative verify step for GB300 (sm_103a).

The product is the C-ABI CUDA library built from ``csrc/`` (see
``include/spec_verify.h``); ``abi`` is its thin ctypes binding, ``runtime``
the PyTorch device-memory plumbing, ``synth`` the seeded synthetic inputs.
Importing this package loads nothing; the library is loaded on first use and
a missing library raises instead of falling back to anything else.
"""
__all__ = ["abi", "runtime", "synth", "build"]
