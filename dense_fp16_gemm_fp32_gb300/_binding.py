"""ctypes binding of libgemm_sm103.so (include/gemm_sm103.h).

Argument marshalling only: tensors are checked and turned into device
pointers, extents and the current CUDA stream; every step of the GEMM runs in
the library's kernels. There is no fallback: if the library is missing or the
tensors are not on a CUDA device, the call raises.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

from . import _build

GEMM_OK = 0
GEMM_ERR_INVALID_ARG = 1
GEMM_ERR_UNSUPPORTED = 2
GEMM_ERR_CUDA = 3
GEMM_ERR_TIMEOUT = 4

TILE_AUTO = 0
TILE_128x256x64 = 1
TILE_128x64x32 = 2
TILE_256x256x64_PAIR = 3
TILE_256x256x128_PAIR = 4
TILE_128x128x64 = 5
TILE_128x128x64_SPLITK = 6
TILE_128x64x64 = 7
TILE_256x256x128_PAIR_ALIGNED = 8
TILE_256x256x64_PAIR_STREAMK = 9
TILE_64x64x64 = 10
TILE_COUNT = 11

DEFAULT_GROUP_SIZE_M = 8

HEADER = os.path.join(_build.ROOT, "include", "gemm_sm103.h")
HEADERS = [HEADER, os.path.join(_build.ROOT, "include", "softmax_sm103.h")]


class GemmError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {status_string(code)} (code {code})")


_lib = None

_c_void_p = ctypes.c_void_p
_SIGNATURES = {
    "gemm_f16_f32acc": (ctypes.c_int, [_c_void_p, _c_void_p, _c_void_p, ctypes.c_int64, ctypes.c_int64,
                                       ctypes.c_int64, ctypes.c_int32, _c_void_p]),
    "gemm_f16_f32acc_tiled": (ctypes.c_int, [_c_void_p, _c_void_p, _c_void_p, ctypes.c_int64, ctypes.c_int64,
                                             ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, _c_void_p,
                                             _c_void_p]),
    "gemm_f16_f32acc_strided": (ctypes.c_int, [_c_void_p, ctypes.c_int64, _c_void_p, ctypes.c_int64, _c_void_p,
                                               ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                               ctypes.c_int32, ctypes.c_int32, _c_void_p, _c_void_p]),
    "gemm_tile_shape": (ctypes.c_int, [ctypes.c_int32, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                       _c_void_p, _c_void_p, _c_void_p]),
    "gemm_tile_config": (ctypes.c_int, [ctypes.c_int32, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, _c_void_p]),
    "gemm_tile_schedule": (ctypes.c_int, [ctypes.c_int64, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                          ctypes.c_int32, _c_void_p, _c_void_p, _c_void_p]),
    "gemm_tile_map_host": (ctypes.c_int, [ctypes.c_int64, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                          ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, _c_void_p, _c_void_p]),
    "gemm_query_status": (ctypes.c_int, [_c_void_p]),
    "gemm_launch_plan": (ctypes.c_int, [ctypes.c_int32, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                        _c_void_p, _c_void_p, _c_void_p]),
    "gemm_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "gemm_last_cuda_error": (ctypes.c_int, []),
    "gemm_set_watchdog_ns": (ctypes.c_int, [ctypes.c_uint64]),
    "gemm_set_fault_injection": (ctypes.c_int, [ctypes.c_int32]),
    "gemm_launch_count": (ctypes.c_uint64, []),
    "gemm_f16_f32acc_noalloc": (ctypes.c_int, [_c_void_p, _c_void_p, _c_void_p, ctypes.c_int64, ctypes.c_int64,
                                               ctypes.c_int64, ctypes.c_int32, _c_void_p, _c_void_p]),
    "gemm_workspace_bytes": (ctypes.c_int, [_c_void_p, ctypes.c_int64, _c_void_p, ctypes.c_int64, _c_void_p,
                                            ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                            _c_void_p]),
    "gemm_f16_f32acc_strided_ws": (ctypes.c_int, [_c_void_p, ctypes.c_int64, _c_void_p, ctypes.c_int64, _c_void_p,
                                                  ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                                  ctypes.c_int32, ctypes.c_int32, _c_void_p, _c_void_p,
                                                  ctypes.c_uint64, _c_void_p]),
    "gemm_autotune": (ctypes.c_int, [_c_void_p, ctypes.c_int64, _c_void_p, ctypes.c_int64, _c_void_p, ctypes.c_int64,
                                     ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                     _c_void_p, _c_void_p, _c_void_p]),
    "gemm_autotune_clear": (ctypes.c_int, []),
    "softmax_rows_f32": (ctypes.c_int, [_c_void_p, ctypes.c_int64, _c_void_p, ctypes.c_int64, ctypes.c_int64,
                                        ctypes.c_int64, _c_void_p]),
    "softmax_rows_plan": (ctypes.c_int, [ctypes.c_int64, ctypes.c_int64, _c_void_p, _c_void_p, _c_void_p]),
    "softmax_launch_count": (ctypes.c_uint64, []),
}

SOFTMAX_MAX_COLS = 65536


def lib_path() -> str:
    return _build.LIB


def load():
    """The loaded library. Raises if it has not been built."""
    global _lib
    if _lib is None:
        path = lib_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with dense_fp16_gemm_fp32_gb300.build() (needs nvcc); "
                "there is no fallback implementation")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def header_functions() -> list[str]:
    """Names of the functions include/gemm_sm103.h and include/softmax_sm103.h declare."""
    names = []
    for path in HEADERS:
        with open(path) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*((?:gemm|softmax)_\w+)\s*\(", text, flags=re.M)
    return names


def status_string(code: int) -> str:
    try:
        return load().gemm_status_string(int(code)).decode()
    except RuntimeError:
        return f"status {code}"


def _check(rc: int, what: str):
    if rc != GEMM_OK:
        raise GemmError(rc, what)


def _stream_ptr(device: torch.device):
    return torch.cuda.current_stream(device).cuda_stream


# The current stream's handle and the current device as plain ints, read from
# torch's C layer without building Python Stream/device objects (a few
# microseconds per call otherwise); the public calls when these are absent.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)
_raw_device = getattr(torch._C, "_cuda_getDevice", None)


def _stream_of(index: int) -> int:
    if _raw_stream is not None:
        return int(_raw_stream(index))
    return torch.cuda.current_stream(index).cuda_stream


def _current_device() -> int:
    return int(_raw_device()) if _raw_device is not None else torch.cuda.current_device()


class _Nothing:
    def __enter__(self):
        return None

    def __exit__(self, *exc):
        return False


_NOTHING = _Nothing()


def _on_device(device: torch.device):
    """torch.cuda.device(device), skipped when it is already current (the
    switch costs microseconds per call)."""
    if device.index is None or device.index == torch.cuda.current_device():
        return _NOTHING
    return torch.cuda.device(device)


def _check_operand(t: torch.Tensor, name: str):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != torch.float16:
        raise TypeError(f"{name} must be float16, got {t.dtype}")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be on a CUDA device, got {t.device}")
    if t.dim() != 2:
        raise ValueError(f"{name} must be 2-D, got shape {tuple(t.shape)}")
    if not _row_major(t):
        raise ValueError(f"{name} must be row-major: unit column stride and a row stride >= its columns")


def _row_major(t: torch.Tensor) -> bool:
    """Row-major, possibly with padded rows: stride (ld, 1) with ld >= columns."""
    rows, cols = t.shape
    if rows <= 1 or cols <= 1:
        return t.is_contiguous() or (t.stride(1) == 1 or cols <= 1)
    return t.stride(1) == 1 and t.stride(0) >= cols


def _ld(t: torch.Tensor) -> int:
    """Row pitch in elements. A one-row tensor's pitch is never used to
    address memory, so it is reported as its row length rounded up to 8."""
    if t.shape[0] > 1:
        return int(t.stride(0))
    return max(8, -(-int(t.shape[1]) // 8) * 8)


def _matrix(t, name: str, dtype=torch.float16):
    """(rows, cols, data pointer, row pitch, device index) of a 2-D row-major
    CUDA matrix, with the checks of _check_operand in one pass."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {str(dtype).replace('torch.', '')}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device, got {t.device}")
    if t.dim() != 2:
        raise ValueError(f"{name} must be 2-D, got shape {tuple(t.shape)}")
    rows, cols = t.shape
    s0, s1 = t.stride()
    if rows > 1 and cols > 1:
        if s1 != 1 or s0 < cols:
            raise ValueError(f"{name} must be row-major: unit column stride and a row stride >= its columns")
    elif not (t.is_contiguous() or s1 == 1 or cols <= 1):
        raise ValueError(f"{name} must be row-major: unit column stride and a row stride >= its columns")
    ld = int(s0) if rows > 1 else max(8, -(-int(cols) // 8) * 8)
    return rows, cols, t.data_ptr(), ld, t.get_device()


def gemm(a: torch.Tensor, b: torch.Tensor, group_size_m: int = DEFAULT_GROUP_SIZE_M,
         out: torch.Tensor | None = None, tile_cfg: int = TILE_AUTO,
         trace: torch.Tensor | None = None, repack: bool = True) -> torch.Tensor:
    """C = a @ b with fp16 operands, fp32 accumulation and one fp16 rounding.

    a: [M,K] fp16 CUDA row-major; b: [K,N] fp16 CUDA row-major, same device.
    Row-major views with padded rows (stride (ld, 1), ld >= columns) are
    accepted with any pitch: pitches that are multiples of 8 elements with
    16-byte aligned data run the TMA kernels in place. Other operands are
    copied into a workspace allocated here (repack=True, the default) and
    the TMA kernels run on the copies; with repack=False they run through
    the library's plain-load kernel instead.
    out: optional [M,N] fp16 CUDA row-major tensor (or padded view) to write;
    its padding columns are not touched.
    trace: optional int32 CUDA tensor of 3 * num_tiles entries that receives
    (pid_m, pid_n, cta) per program id, as the kernel's scheduler ran them.
    Runs on the current CUDA stream of a's device.
    """
    M, K, pa, lda, dev_a = _matrix(a, "a")
    K2, N, pb, ldb, dev_b = _matrix(b, "b")
    if dev_a != dev_b:
        raise ValueError("a and b must be on the same device")
    if K != K2:
        raise ValueError(f"inner extents differ: a is {tuple(a.shape)}, b is {tuple(b.shape)}")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=a.device)
        pc, ldc = out.data_ptr(), (N if M > 1 else max(8, -(-N // 8) * 8))
    else:
        Mo, No, pc, ldc, dev_c = _matrix(out, "out")
        if (Mo, No) != (M, N) or dev_c != dev_a:
            raise ValueError(f"out must be [{M},{N}] on {a.device}")
    lib = _lib if _lib is not None else load()
    args = (pa, lda, pb, ldb, pc, ldc, M, N, K)
    # operands that already suit the tensor maps need no workspace query
    tma_shaped = (pc | (pa | pb if K else 0)) & 15 == 0 and (ldc | (lda | ldb if K else 0)) & 7 == 0
    trace_ptr = None
    if trace is not None:
        if trace.dtype != torch.int32 or trace.device != a.device or not trace.is_contiguous():
            raise ValueError("trace must be a contiguous int32 tensor on a's device")
        tm, tn, _ = tile_shape(tile_cfg, M, N, K)
        tiles = -(-M // tm) * -(-N // tn)
        if not tma_shaped and not repack:  # the generic-load kernel's 128 x 256 tiles
            tiles = max(tiles, -(-M // 128) * -(-N // 256))
        if trace.numel() < 3 * tiles:
            raise ValueError(f"trace needs {3 * tiles} entries (3 per tile), got {trace.numel()}")
        trace_ptr = trace.data_ptr()
    if tma_shaped and dev_a == _current_device():  # the common case: no workspace, no device switch
        rc = lib.gemm_f16_f32acc_strided(*args, int(group_size_m), int(tile_cfg), trace_ptr, _stream_of(dev_a))
        if rc != GEMM_OK:
            raise GemmError(rc, "gemm_f16_f32acc_strided")
        return out
    dev = a.device
    with _on_device(dev):
        need = ctypes.c_uint64(0)
        if repack and not tma_shaped:
            _check(lib.gemm_workspace_bytes(*args, ctypes.byref(need)), "gemm_workspace_bytes")
        stream = _stream_of(dev_a)
        if need.value:
            ws = torch.empty(need.value, dtype=torch.uint8, device=dev)  # caching allocator: stream-ordered reuse
            rc = lib.gemm_f16_f32acc_strided_ws(*args, int(group_size_m), int(tile_cfg), trace_ptr, ws.data_ptr(),
                                                need.value, stream)
            _check(rc, "gemm_f16_f32acc_strided_ws")
        else:
            rc = lib.gemm_f16_f32acc_strided(*args, int(group_size_m), int(tile_cfg), trace_ptr, stream)
            _check(rc, "gemm_f16_f32acc_strided")
    return out


def tile_shape(tile_cfg: int = TILE_AUTO, M: int = 0, N: int = 0, K: int = 0) -> tuple[int, int, int]:
    tm, tn, tk = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    _check(load().gemm_tile_shape(int(tile_cfg), M, N, K, ctypes.byref(tm), ctypes.byref(tn), ctypes.byref(tk)),
           "gemm_tile_shape")
    return tm.value, tn.value, tk.value


def tile_config(tile_cfg: int = TILE_AUTO, M: int = 0, N: int = 0, K: int = 0) -> int:
    """The configuration tile_cfg resolves to for (M, N, K) (TILE_AUTO: the tuned or rule choice)."""
    r = ctypes.c_int32()
    _check(load().gemm_tile_config(int(tile_cfg), M, N, K, ctypes.byref(r)), "gemm_tile_config")
    return r.value


def launch_plan(M: int, N: int, K: int = 0, tile_cfg: int = TILE_AUTO, device=None) -> dict:
    """How the library schedules a problem on a device: grid CTAs, tiles, split tail tiles."""
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    ctas, tiles, split = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    with torch.cuda.device(device):
        rc = load().gemm_launch_plan(int(tile_cfg), M, N, K, ctypes.byref(ctas), ctypes.byref(tiles),
                                     ctypes.byref(split))
    _check(rc, "gemm_launch_plan")
    return {"grid_ctas": ctas.value, "num_tiles": tiles.value, "split_tiles": split.value}


def tile_schedule(M: int, N: int, tile_m: int, tile_n: int, group_size_m: int, device=None):
    """(pid_m, pid_n) int32 CUDA tensors of the device-side grouped map."""
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    n = -(-M // tile_m) * -(-N // tile_n) if M > 0 and N > 0 else 0
    pm = torch.empty(max(n, 1), dtype=torch.int32, device=device)
    pn = torch.empty(max(n, 1), dtype=torch.int32, device=device)
    with torch.cuda.device(device):
        rc = load().gemm_tile_schedule(M, N, tile_m, tile_n, group_size_m, pm.data_ptr(), pn.data_ptr(),
                                       _stream_ptr(device))
    _check(rc, "gemm_tile_schedule")
    return pm[:n], pn[:n]


def tile_map_host(M: int, N: int, tile_m: int, tile_n: int, group_size_m: int, pid0: int = 0, count=None):
    """(pid_m, pid_n) int32 numpy arrays of the kernels' grouped map evaluated on the host
    for pids [pid0, pid0 + count) (default: every tile). Needs no GPU."""
    import numpy as np

    n = -(-M // tile_m) * -(-N // tile_n) if M > 0 and N > 0 else 0
    count = n - pid0 if count is None else count
    pm = np.zeros(max(count, 1), dtype=np.int32)
    pn = np.zeros(max(count, 1), dtype=np.int32)
    rc = load().gemm_tile_map_host(M, N, tile_m, tile_n, group_size_m, pid0, count, pm.ctypes.data, pn.ctypes.data)
    _check(rc, "gemm_tile_map_host")
    return pm[:count], pn[:count]


def query_status(device=None) -> int:
    """Synchronise the current stream and return (and clear) the device status."""
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(device):
        return int(load().gemm_query_status(_stream_ptr(device)))


def set_watchdog_ns(ns: int) -> None:
    _check(load().gemm_set_watchdog_ns(int(ns)), "gemm_set_watchdog_ns")


def set_fault_injection(mode: int) -> None:
    _check(load().gemm_set_fault_injection(int(mode)), "gemm_set_fault_injection")


def launch_count() -> int:
    return int(load().gemm_launch_count())


def last_cuda_error() -> int:
    return int(load().gemm_last_cuda_error())


def _check_rows(t: torch.Tensor, name: str):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != torch.float32:
        raise TypeError(f"{name} must be float32, got {t.dtype}")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be on a CUDA device, got {t.device}")
    if t.dim() != 2:
        raise ValueError(f"{name} must be 2-D, got shape {tuple(t.shape)}")
    if not _row_major(t):
        raise ValueError(f"{name} must be row-major: unit column stride and a row stride >= its columns")


def _row_pitch(t: torch.Tensor) -> int:
    """Row pitch in elements; a one-row tensor's pitch addresses nothing and
    is reported as its row length rounded up to 4."""
    if t.shape[0] > 1:
        return int(t.stride(0))
    return max(4, -(-int(t.shape[1]) // 4) * 4)


def softmax(x: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
    """Row softmax of x along dim 1 (fp32), as the fused-softmax tutorial computes it.

    x: [M, n] fp32 CUDA, row-major; a view with padded rows (stride (ld, 1),
    ld >= n) is read in place and its padding is not read.
    out: optional [M, n] fp32 CUDA row-major tensor or padded view (may be x
    itself); its padding columns are not written. By default the result is a
    [M, n] view of a new array whose rows are padded to a multiple of 4
    elements, so that every row starts on a 16-byte boundary.
    Runs on the current CUDA stream of x's device.
    """
    _check_rows(x, "x")
    M, n = x.shape
    if out is None:
        ld = max(4, -(-n // 4) * 4)
        out = torch.empty((M, ld), dtype=torch.float32, device=x.device)[:, :n]
    else:
        _check_rows(out, "out")
        if tuple(out.shape) != (M, n) or out.device != x.device:
            raise ValueError(f"out must be [{M},{n}] on {x.device}")
    lib = _lib if _lib is not None else load()
    with _on_device(x.device):
        rc = lib.softmax_rows_f32(x.data_ptr(), _row_pitch(x), out.data_ptr(), _row_pitch(out), M, n,
                                  _stream_ptr(x.device))
    _check(rc, "softmax_rows_f32")
    return out


def softmax_plan(M: int, n: int, device=None) -> dict:
    """The launch softmax() makes for M rows of n columns: threads and CTAs per row, grid CTAs."""
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    tpr, cl, grid = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    with torch.cuda.device(device):
        rc = load().softmax_rows_plan(M, n, ctypes.byref(tpr), ctypes.byref(cl), ctypes.byref(grid))
    _check(rc, "softmax_rows_plan")
    return {"threads_per_row": tpr.value, "cluster_ctas": cl.value, "grid_ctas": grid.value}


def softmax_launch_count() -> int:
    return int(load().softmax_launch_count())


def workspace_bytes(a: torch.Tensor, b: torch.Tensor, out: torch.Tensor) -> int:
    """Workspace gemm() allocates for these operands (0 when all suit the TMA kernels)."""
    need = ctypes.c_uint64(0)
    M, K = a.shape
    N = b.shape[1]
    _check(load().gemm_workspace_bytes(a.data_ptr(), _ld(a), b.data_ptr(), _ld(b), out.data_ptr(), _ld(out), M, N, K,
                                       ctypes.byref(need)), "gemm_workspace_bytes")
    return int(need.value)


def autotune(a: torch.Tensor, b: torch.Tensor, out: torch.Tensor | None = None,
             group_size_m: int = DEFAULT_GROUP_SIZE_M, reps: int = 20) -> dict:
    """Times every tile configuration on a @ b (out is overwritten) and makes
    the fastest the TILE_AUTO choice for this shape on this device.
    Returns {"best": cfg, "us": {cfg: microseconds per launch}} (configurations
    that do not apply to the shape, such as the aligned one on partial tiles,
    are left out)."""
    _check_operand(a, "a")
    _check_operand(b, "b")
    if a.device != b.device:
        raise ValueError("a and b must be on the same device")
    M, K = a.shape
    K2, N = b.shape
    if K != K2:
        raise ValueError(f"inner extents differ: a is {tuple(a.shape)}, b is {tuple(b.shape)}")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=a.device)
    else:
        _check_operand(out, "out")
        if tuple(out.shape) != (M, N) or out.device != a.device:
            raise ValueError(f"out must be [{M},{N}] on {a.device}")
    best = ctypes.c_int32(0)
    us = (ctypes.c_float * TILE_COUNT)()
    with _on_device(a.device):
        rc = load().gemm_autotune(a.data_ptr(), _ld(a), b.data_ptr(), _ld(b), out.data_ptr(), _ld(out), M, N, K,
                                  int(group_size_m), int(reps), ctypes.byref(best), us,
                                  _stream_ptr(a.device))
    _check(rc, "gemm_autotune")
    return {"best": best.value, "us": {c: float(us[c]) for c in range(1, TILE_COUNT) if us[c] >= 0}}


def autotune_clear() -> None:
    _check(load().gemm_autotune_clear(), "gemm_autotune_clear")
