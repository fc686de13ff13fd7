"""GB300-native ring all-reduce of N virtual ranks held in one GPU's memory.

The CUDA library (``libra.so``, built from ``csrc/``) does all the work; the
Python binding in ``ring_all_reduce_02_gb300.ra`` only marshals arguments.
Importing this package does not load the library; the first call does, and
fails loudly if it is missing.
"""

__all__ = ["ra", "inputs"]
