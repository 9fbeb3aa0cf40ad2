"""Gated DeltaNet token-mixing path on GB300 (sm_103a).

The compute lives in ``libgdn.so`` (hand-written CUDA kernels behind a C ABI,
declared in ``include/gdn.h``); :mod:`.gdn` is the thin ctypes binding with the
same entry-point names. :mod:`.synthetic` generates seeded inputs.
"""
