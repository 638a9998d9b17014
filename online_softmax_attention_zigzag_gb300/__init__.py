"""GB300-native (sm_103a) per-rank hot path of ring attention with zigzag chunking.

The compute runs in hand-written CUDA kernels behind the C ABI of
``libringattn.so`` (declared in ``include/ringattn.h``); :mod:`.ringattn` is
the thin Python binding that the tests and the benchmark call.
"""
