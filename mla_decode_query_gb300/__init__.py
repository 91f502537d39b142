"""GB300-native fused MLA decode query projection and assembly (and the V
up-projection after attention).

The operation runs in ``libmlaqp.so`` (CUDA C++ for sm_103a, C ABI in
``include/mlaqp.h``); ``mla_decode_query_gb300.mlaqp`` is its thin ctypes
binding and ``mla_decode_query_gb300.inputs`` the seeded synthetic inputs.
Importing the package does not load the library; the first call does, and
fails loudly if it has not been built.
"""

from .mlaqp import (  # noqa: F401
    ARMS,
    MAX_M,
    MAX_M_DECODE,
    V_HEAD_DIM,
    MLAQP_DEVSTATUS_WAIT_TIMEOUT,
    MLAQP_ERR_CUDA,
    MLAQP_ERR_INVALID_ARG,
    MLAQP_ERR_UNSUPPORTED,
    MLAQP_OK,
    MLAQP_OUT_BF16,
    MLAQP_OUT_E4M3,
    MLAQP_WEIGHT_BF16,
    MLAQP_WEIGHT_MXFP8,
    MlaqpError,
    check,
    header_functions,
    load_library,
    mlaqp_can_implement,
    mlaqp_debug_launch_null,
    mlaqp_debug_plan,
    mlaqp_debug_run_arm,
    mlaqp_debug_set_policy,
    mlaqp_debug_run_bounded_wait,
    mlaqp_debug_v_plan,
    mlaqp_debug_v_up_bounded_wait,
    mlaqp_device_status,
    mlaqp_last_error,
    mlaqp_launch_shape,
    mlaqp_prefetch_weights,
    mlaqp_prewarm,
    mlaqp_run,
    mlaqp_run_pdl,
    mlaqp_run_strided,
    mlaqp_v_up_can_implement,
    mlaqp_v_up_prewarm,
    mlaqp_v_up_run,
    mlaqp_version,
)

__version__ = "0.1.0"
