"""GB300-native paged-KV decode attention.

The compute path is the C-ABI library built from csrc/ (hand-written CUDA for
sm_103a); this package holds the ctypes binding to it and the seeded input
generator. Importing the package does not load the library; the first call
does, and fails loudly if it is missing.
"""

__all__ = ["inputs"]
