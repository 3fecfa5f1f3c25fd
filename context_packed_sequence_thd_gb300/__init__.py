"""GB300-native context-parallel causal attention over THD-packed documents.

The compute path lives in ``libcpthd.so`` (hand-written sm_103a CUDA behind a
C ABI declared in ``include/cpthd.h``); :mod:`.api` is a thin ctypes binding
with the same names.  The binding is loaded lazily so that the input
generators in :mod:`.inputs` import on machines without the built library.
"""
__version__ = "0.1.0"
