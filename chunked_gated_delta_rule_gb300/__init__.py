"""GB300-native chunked gated-delta-rule forward pass.

The compute path is a C-ABI CUDA library (``include/gdr.h``); this package is
its thin ctypes binding plus the seeded synthetic input generator.
"""
