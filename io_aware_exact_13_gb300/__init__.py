"""Exact IO-aware tiled attention forward for GB300 (sm_103a).

The compute path is the C-ABI library ``libfa.so`` built from ``csrc/``; the
Python binding in ``fa.py`` only marshals pointers, sizes and the CUDA stream.
``inputs.py`` draws seeded synthetic inputs. Importing this package does not
load the library: ``from io_aware_exact_13_gb300 import fa`` does, and fails
loudly when it has not been built.
"""
__all__ = ["fa", "inputs", "build"]
__version__ = "0.1.0"
