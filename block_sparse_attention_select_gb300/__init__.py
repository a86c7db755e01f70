"""GB300-native QSA indexer: paged FP16 index scoring + exact top-k (sm_103a).

The compute lives in a C-ABI shared library (``libqsa.so``, built from
``csrc/``); :mod:`.qsa` is the thin ctypes binding with the same entry-point
names, and :mod:`.workloads` draws seeded synthetic inputs.  Importing this
package does not load the library; the binding loads it on first use and
raises if it is missing.
"""
__all__ = ["qsa", "workloads"]
