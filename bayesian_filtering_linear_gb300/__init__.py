"""GB300-native Kalman Linear Attention scan.

The compute path is the C-ABI library ``libkla.so`` (hand-written sm_103a
CUDA); :mod:`bayesian_filtering_linear_gb300.kla` is its thin ctypes binding.
:mod:`bayesian_filtering_linear_gb300.inputs` draws seeded synthetic inputs.
"""
