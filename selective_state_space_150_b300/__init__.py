"""libssmscan: the selective-scan forward pass of the Mamba S6 layer on B300.

The computation lives in the CUDA library ``libssmscan.so`` (C ABI declared in
``include/ssmscan.h``); ``ssmscan`` is its thin Python binding.
"""
from .ssmscan import (  # noqa: F401
    SSMError,
    conv_selective_scan_fwd,
    selective_scan_bwd,
    selective_scan_fwd,
    selective_scan_step,
    ssm_conv_scan_fwd,
    ssm_conv_scan_fwd_bf16,
    ssm_scan_bwd,
    ssm_scan_bwd_bf16,
    ssm_scan_bwd_bf16_h0,
    ssm_scan_bwd_h0,
    ssm_scan_fwd,
    ssm_scan_fwd_bf16,
    ssm_scan_fwd_bf16_host,
    ssm_scan_fwd_host,
    ssm_scan_host_workspace_bytes,
    ssm_scan_fwd_bf16_noalloc,
    ssm_scan_fwd_bf16_h0,
    ssm_scan_fwd_bf16_zoh,
    ssm_scan_fwd_h0,
    ssm_scan_fwd_zoh,
    ssm_scan_step,
    ssm_scan_step_bf16,
    ssm_scan_last_device_status,
    ssm_scan_plan,
    ssm_set_knob,
    ssm_status_string,
)
