"""GB300-native SnapKV observation-window KV-cache selection.

The compute lives in the CUDA library ``libkvsel.so`` (C ABI declared in
``include/kvsel.h``); ``api`` is a thin ctypes binding with the same names.
Importing this package does not load the library; the first API call does,
and raises if the library is missing.
"""

__all__ = ["api", "workloads"]
