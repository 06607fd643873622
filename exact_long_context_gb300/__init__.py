"""Exact long-context attention on one GB300 (sm_103a).

The compute path is the C-ABI library ``libra.so`` built from ``csrc/``; the Python
module :mod:`exact_long_context_gb300.ra` marshals torch tensors into its calls.
Importing this package loads nothing; the library is loaded on first use and its
absence is an error (there is no CPU fallback).
"""

__all__ = ["ra", "synth"]
