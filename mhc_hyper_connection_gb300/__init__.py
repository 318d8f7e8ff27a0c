"""GB300 (sm_103a) mHC pre-mapping forward and backward, and the post-mapping:
C ABI + thin ctypes binding.

The compute lives in ``libmhc_pre.so`` (built from ``csrc/`` by
``python -m mhc_hyper_connection_gb300.build``).  This package only loads it
and marshals arguments; importing it does not load the library until a
function is called.
"""
from ._binding import (  # noqa: F401
    LAUNCH_FIELDS, LIB_PATH, MHC_DTYPE_BF16, MHC_DTYPE_FP16, MHC_KERNEL_AUTO, MHC_KERNEL_CLUSTER, MHC_KERNEL_GRID, MHC_KERNEL_RESIDENT, MHC_ERR_NULLPTR, MHC_ERR_PARAM_INVALID, MHC_ERR_RUNTIME, MHC_IMPL_FP32,
    MHC_IMPL_TF32, MHC_OK, MhcError, MhcPre, MhcPreArgs, MhcPreBwdArgs, MhcPreConfig, hc_post, last_error,
    library, mhc_post_run, mhc_pre_backward_run, mhc_pre_backward_workspace_size, mhc_pre_inv_rms_run,
    mhc_pre_mixes_run, mhc_pre_sinkhorn_run,
    mhc_pre_config_default, mhc_pre_create, mhc_pre_destroy, mhc_pre_last_kernel, mhc_pre_last_launch, mhc_pre_run, mhc_pre_run_noalloc, mhc_pre_set_profile_events, mhc_pre_set_wait_test, mhc_pre_status, mhc_pre_weights_size, mhc_pre_prepare_weights,
    mhc_pre_workspace_size, status_string)
