"""libkbattn: scaled-dot-product attention forward for GB300 (sm_103a).

The compute path is the C-ABI shared library ``libkbattn.so`` built from
``csrc/``; ``kbattn`` is its thin ctypes binding. Importing this package does
not load the library; ``kbattn.load()`` (or the first call) does, and fails
loudly if it has not been built.
"""
__all__ = ["inputs", "kbattn", "roofline"]
