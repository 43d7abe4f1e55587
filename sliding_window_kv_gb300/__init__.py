"""sliding_window_kv_gb300: incremental sliding-window KV attention on one GB300.

The product is the C-ABI library ``libvst.so`` (``include/vst.h``) built from ``csrc/`` by
``build.py``; ``vst`` is its thin Python binding and ``synth`` the seeded input generator.
Importing the package loads nothing; the library is loaded on first use.
"""
__all__ = ["vst", "synth", "build"]
