"""Gated delta-rule recurrence (Gated DeltaNet) for one GB300, sm_103a.

The compute path is the C-ABI library ``libgdn.so`` (hand-written CUDA);
``gated_deltanet_recurrence_02_gb300.gdn`` is its thin ctypes binding, with
the same entry-point names as ``include/gdn.h``.  ``inputs`` draws the seeded
synthetic workloads.  Importing the package loads nothing; the first call
into ``gdn`` loads the library and raises if it is missing.
"""
__all__ = ["gdn", "inputs"]
