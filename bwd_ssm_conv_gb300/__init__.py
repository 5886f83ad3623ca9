"""GB300 (sm_103a) selective state-space scan with its causal depthwise conv1d prelude.

The compute lives in ``libssm_gb300.so`` (hand-written CUDA behind the C ABI of
``include/ssm.h``); this package is a thin ctypes binding with the same entry-point names.
PyTorch supplies device memory and streams only.
"""
