"""B300-native Introspective Strided Decoding (ISD) verify-and-propose step.

The step runs in hand-written CUDA kernels for sm_103a behind a C ABI
(``include/isd.h``); :mod:`.isd` is the thin ctypes binding with the same
names.  The native library is loaded on first use and its absence is an
error: there is no CPU fallback.
"""
