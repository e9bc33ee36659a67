"""GB300-native (sm_103a) attention-KL primitive: KL(P1 || P2) between a
teacher and a student attention distribution per query row, with gradients,
without materialising the N_Q x N_K score or probability matrices.

The computation lives in the CUDA library built from ``csrc/`` (C ABI in
``include/streamkl.h``); this package only marshals arguments to it.
"""
from .binding import (  # noqa: F401
    BWD_FUSED,
    BWD_SEPARATE,
    STREAMKL_ERR_CUDA,
    STREAMKL_ERR_DEVICE_CHECK,
    STREAMKL_ERR_INVALID_ARG,
    STREAMKL_ERR_TIMEOUT,
    STREAMKL_ERR_UNSUPPORTED,
    STREAMKL_OK,
    StreamKLError,
    bwd_algorithm,
    bwd_dk_persist,
    bwd_dq_splits,
    choose_splits,
    fwd_pairs,
    load,
    new_status,
    raise_on_device_status,
    selftest_device_check,
    selftest_wait_timeout,
    set_bwd_algorithm,
    set_bwd_dk_persist,
    set_bwd_dq_splits,
    set_fwd_pairs,
    use_debug_library,
    streamkl_bwd,
    streamkl_bwd_reverse,
    streamkl_bwd_varlen,
    streamkl_bwd_workspace_size,
    streamkl_fwd,
    streamkl_fwd_reverse,
    streamkl_fwd_noalloc,
    streamkl_fwd_varlen,
    streamkl_fwd_workspace_size,
    streamkl_workspace_size,
)

__version__ = "0.2.0"
