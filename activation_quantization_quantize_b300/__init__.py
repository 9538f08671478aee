"""B300-native quantized linear layer: affine quantizer, W8A8 and W4A16 GEMMs.

The compute lives in ``libqlin.so`` (hand-written CUDA for sm_103a behind the C
ABI of ``include/qlin.h``); :mod:`.qlin` is its ctypes binding and
:mod:`.inputs` draws the seeded synthetic workloads.
"""
