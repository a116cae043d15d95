"""GB300-native hot path of QSpec-style quantized speculative decoding.

The compute lives in ``libqspec.so`` (CUDA for sm_103a, C ABI in include/qspec.h); ``qspec`` is
its ctypes binding; ``synthetic`` draws the seeded inputs.
"""
