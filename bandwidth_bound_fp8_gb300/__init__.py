"""bandwidth_bound_fp8_gb300: the FP8 live-quantised MoE expert projection
for small decode batches on GB300, as the C-ABI library libmoeq.so plus the
thin Python binding in ``moeq``.

Build the library with ``python -m bandwidth_bound_fp8_gb300.build`` (or
``__graft_entry__.build()``); importing ``bandwidth_bound_fp8_gb300.moeq``
and calling any function loads it and raises if it is missing.
"""
from . import moeq  # noqa: F401

__all__ = ["moeq"]
