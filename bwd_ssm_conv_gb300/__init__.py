"""GB300 (sm_103a) selective state-space scan with its causal depthwise conv1d prelude.

The compute lives in ``libssm_gb300.so`` (hand-written CUDA behind the C ABI of
``include/ssm.h``); ``binding`` is a thin ctypes layer with the same entry-point names.
PyTorch supplies device memory and streams only.
"""
from .binding import (  # noqa: F401
    GRAD_NAMES, SsmError, ScanShape, lib, pack_conv_grads, pack_scan_grads, pack_scan_result,
    scan_shape, ssm_abi_version, ssm_kernel_launches, ssm_conv_bwd, ssm_conv_fwd, ssm_conv_workspace_size,
    ssm_decode_step, ssm_scan_bwd, ssm_scan_fwd, ssm_scan_status, ssm_scan_workspace_size,
    ssm_status_string,
)
