"""GB300-native selective state-space scan: a C-ABI CUDA library (``libssm.so``)
and its thin Python binding.

Entry points (same names as in ``include/ssm.h``): ``ssm_scan_fwd``,
``ssm_scan_bwd``, ``ssm_scan_fwd_host``, ``ssd_chunked_fwd``, ``ssd_chunked_bwd``, ``ssm_decode_step``, ``ssd_mamba3_fwd``,
``ssm_decode_step_mamba3``, ``ssd_mamba3_mimo_fwd``, ``ssm_decode_step_mamba3_mimo``,
``ssm_scan_workspace_bytes``, ``ssm_scan_bwd_workspace_bytes``,
``ssm_last_device_status``.  The library is loaded on first call; building it is
``state_space_model_selective_gb300.build.build()``.
"""
from .binding import (EXPORTS, SSMError, lib, ssd_chunked_bwd,  # noqa: F401
                      ssd_chunked_checkpoint_bytes,
                      ssd_chunked_bwd_workspace_bytes, ssd_chunked_fwd, ssd_mamba3_fwd,
                      ssd_mamba3_mimo_fwd, ssm_abi_version, ssm_decode_step,
                      ssm_decode_step_mamba3, ssm_decode_step_mamba3_mimo,
                      ssm_last_device_status, ssm_scan_bwd, ssm_scan_bwd_workspace_bytes,
                      ssm_scan_checkpoint_bytes, ssm_scan_fwd, ssm_scan_fwd_host,
                      ssm_scan_fwd_host_workspace_bytes,
                      ssm_scan_workspace_bytes, status_string)
