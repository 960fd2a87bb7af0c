"""GB300-native FP32 SGEMM: C = alpha*A*B + beta*C on row-major float32 matrices.

The product runs in hand-written sm_103a CUDA kernels behind the C ABI in
include/sgemm.h (libsgemm_gb300.so, built in-tree by ``build.build()``).
This package is the thin Python binding over that library; the first call
raises if the library has not been built -- there is no CPU or library
fallback.
"""
from ._lib import (  # noqa: F401
    SGEMM_ERR_CUDA,
    SGEMM_ERR_INVALID_ARG,
    SGEMM_ERR_NOMEM,
    SGEMM_ERR_TIMEOUT,
    SGEMM_ERR_UNSUPPORTED,
    SGEMM_OK,
    SGEMM_TUNE_TENSOR_CORES,
    Plan,
    SgemmError,
    autotune,
    clear_plan_cache,
    config_id,
    config_name,
    config_names,
    device_status,
    lib,
    num_configs,
    plan_cache_size,
    probe_ffma,
    run_static_scratch,
    selftest_wait_timeout,
    set_wait_timeout_ns,
    wait_limit_ns,
    table_choice,
    streamk_schedule,
    sgemm,
    status_string,
)
