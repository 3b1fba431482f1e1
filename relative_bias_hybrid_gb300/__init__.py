"""GB300-native (sm_103a) attention hot path of the Inkling decoder layer.

The compute lives in ``libinkattn.so`` (hand-written CUDA behind a C ABI,
declared in ``include/inkattn.h``); ``relative_bias_hybrid_gb300.inkattn``
is the thin ctypes binding with the same entry-point names.
"""
