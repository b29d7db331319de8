"""GB300-native target-side verify step of speculative decoding.

The compute path is the C-ABI library ``libspecdec.so`` (hand-written CUDA for
sm_103a, built from ``csrc/``); this package holds its thin Python binding and
the seeded synthetic input generators (``workloads``).
"""
