"""fp16 GEMM with fp32 accumulation for GB300 (sm_103a), and a fused row softmax.

    C[M,N] = A[M,K] @ B[K,N]   (fp16 in, fp32 accumulate, fp16 out, rounded once)
    Y[i,:] = softmax(X[i,:n])  (fp32, one pass over memory)

The work runs in hand-written CUDA kernels (tcgen05/TMA for the GEMM) behind
a C ABI (include/gemm_sm103.h, include/softmax_sm103.h, libgemm_sm103.so);
this package is its thin Python binding plus the seeded synthetic inputs
used by the tests and the benchmark.
"""
from ._binding import (  # noqa: F401
    DEFAULT_GROUP_SIZE_M,
    GEMM_ERR_CUDA,
    GEMM_ERR_INVALID_ARG,
    GEMM_ERR_TIMEOUT,
    GEMM_ERR_UNSUPPORTED,
    GEMM_OK,
    SOFTMAX_MAX_COLS,
    TILE_128x64x32,
    TILE_128x64x64,
    TILE_64x64x64,
    TILE_128x128x64,
    TILE_128x128x64_SPLITK,
    TILE_128x256x64,
    TILE_256x256x64_PAIR,
    TILE_256x256x128_PAIR,
    TILE_256x256x128_PAIR_ALIGNED,
    TILE_256x256x64_PAIR_STREAMK,
    TILE_AUTO,
    TILE_COUNT,
    GemmError,
    autotune,
    autotune_clear,
    gemm,
    header_functions,
    last_cuda_error,
    launch_count,
    launch_plan,
    lib_path,
    load,
    query_status,
    set_fault_injection,
    set_watchdog_ns,
    softmax,
    softmax_launch_count,
    softmax_plan,
    status_string,
    tile_config,
    tile_map_host,
    tile_schedule,
    tile_shape,
    workspace_bytes,
)
from ._build import build  # noqa: F401
