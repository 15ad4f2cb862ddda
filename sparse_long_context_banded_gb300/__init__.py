"""Banded + global sparse attention (Longformer / GMAT form), forward pass, GB300.

The compute path is the C-ABI CUDA library built from ``csrc/`` (see
``include/sa.h``); ``sa`` is its thin ctypes binding and ``inputs`` holds the
seeded synthetic workloads.  Importing the package does not load the library.
"""
__all__ = ["inputs", "sa"]
