"""GB300-native FP8 (e4m3) GEMM with fine-grained (1x128 / 128x128) scaling.

The compute path is the C-ABI library ``libfp8gemm.so`` built from ``csrc/``
for sm_103a; :mod:`.binding` is the thin ctypes layer over it (argument
marshalling only).  Importing this package does not load the library; the
first call through :mod:`.binding` does, and raises if it is missing.
"""

__all__ = ["binding", "synthetic"]
