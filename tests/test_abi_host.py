"""Host-side checks of the C ABI: the library builds, loads and exports every
function include/gemm_sm103.h declares, and argument validation answers
without a GPU (validation runs before any CUDA call)."""
import ctypes

import pytest
import torch

import dense_fp16_gemm_fp32_gb300 as g


@pytest.fixture(scope="module")
def lib():
    g.build()
    return g.load()


def test_header_declares_expected_entry_points():
    names = g.header_functions()
    for want in ("gemm_f16_f32acc", "gemm_f16_f32acc_tiled", "gemm_tile_schedule", "gemm_query_status",
                 "softmax_rows_f32", "softmax_rows_plan", "softmax_launch_count",
                 "gemm_status_string", "gemm_tile_shape", "gemm_set_watchdog_ns", "gemm_set_fault_injection",
                 "gemm_launch_count", "gemm_last_cuda_error"):
        assert want in names
    assert len(names) == len(set(names))


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(g.lib_path())
    for name in g.header_functions():
        assert hasattr(raw, name), name


def test_status_strings(lib):
    for code in range(5):
        s = g.status_string(code)
        assert s.startswith("GEMM_")
    assert "unknown" in g.status_string(99)


def test_tile_shapes(lib):
    assert g.tile_shape(g.TILE_AUTO, M=128, N=4096, K=512) == (64, 64, 64)       # one band, 128 tiles of 64x64
    assert g.tile_shape(g.TILE_AUTO, M=128, N=8192, K=512) == (128, 64, 64)      # 256 tiles of 64x64: 128x64
    assert g.tile_shape(g.TILE_AUTO, M=128, N=4096, K=1024) == (128, 128, 64)    # one band, 32 tiles: split-K
    assert g.tile_shape(g.TILE_AUTO, M=256, N=2048, K=1024) == (256, 256, 128)   # two bands at K = 1024: pair
    assert g.tile_shape(g.TILE_AUTO, M=128, N=16384, K=1024) == (128, 256, 64)   # one band, 256 tiles of 128x64
    assert g.tile_shape(g.TILE_AUTO, M=129, N=8192, K=1024) == (256, 256, 128)   # 32 pair tiles: all split
    assert g.tile_shape(g.TILE_AUTO, M=129, N=10240, K=1024) == (128, 256, 64)   # 40 pair tiles: under one wave
    assert g.tile_shape(g.TILE_AUTO, M=2048, N=1024, K=512) == (128, 128, 64)    # 32 pair tiles, short K
    assert g.tile_shape(g.TILE_AUTO, M=2048, N=2048, K=2048) == (256, 256, 64)   # 64 pair tiles, K >= 2048
    assert g.tile_shape(g.TILE_AUTO, M=2048, N=2048, K=1024) == (128, 256, 64)   # 64 pair tiles, shorter K
    assert g.tile_config(g.TILE_AUTO, M=2048, N=2048, K=4096) == g.TILE_256x256x64_PAIR  # under a wave: no stream-K
    assert g.tile_shape(g.TILE_AUTO, M=2048, N=2560, K=4096) == (256, 256, 64)   # 80 pair tiles, K <= 4096
    assert g.tile_shape(g.TILE_AUTO, M=2048, N=2560, K=4097) == (256, 256, 64)   # deeper K: 64-deep as well
    assert g.tile_shape(g.TILE_AUTO, M=4096, N=3072, K=256) == (128, 256, 64)    # few k steps
    assert g.tile_shape(g.TILE_AUTO, M=512, N=512, K=512) == (64, 64, 64)        # 64 tiles of 64x64, short K
    assert g.tile_shape(g.TILE_AUTO, M=1024, N=1024, K=512) == (128, 64, 64)     # 128 of them: one wave
    assert g.tile_shape(g.TILE_AUTO, M=1024, N=1024, K=1024) == (256, 256, 128)  # few, long enough K
    assert g.tile_shape(g.TILE_AUTO, M=1024, N=768, K=128) == (128, 64, 64)
    assert g.tile_shape(g.TILE_AUTO, M=1024, N=2048, K=256) == (128, 128, 64)    # 256 tiles of 128x64: two waves
    assert g.tile_shape(g.TILE_AUTO, M=128, N=4096, K=4096) == (128, 128, 64)    # split-K
    assert g.tile_shape(g.TILE_AUTO, M=8192, N=8192, K=8192) == (256, 256, 64)
    assert g.tile_shape(g.TILE_AUTO, M=16384, N=16384, K=16384) == (256, 256, 64)
    # stream-K: 192 pair tiles (a last wave of 40 of 76) with K >= 4096; not for shorter K or many waves
    assert g.tile_config(g.TILE_AUTO, M=4096, N=3072, K=8192) == g.TILE_256x256x64_PAIR_STREAMK
    assert g.tile_config(g.TILE_AUTO, M=4096, N=3072, K=4096) == g.TILE_256x256x64_PAIR_STREAMK
    assert g.tile_config(g.TILE_AUTO, M=4096, N=3072, K=2048) == g.TILE_256x256x64_PAIR
    assert g.tile_config(g.TILE_AUTO, M=4095, N=3000, K=1000) == g.TILE_256x256x64_PAIR
    assert g.tile_config(g.TILE_AUTO, M=8192, N=8192, K=8192) == g.TILE_256x256x64_PAIR    # last wave of 36
    assert g.tile_config(g.TILE_AUTO, M=16384, N=16384, K=16384) == g.TILE_256x256x64_PAIR  # 54 waves
    assert g.tile_config(g.TILE_AUTO, M=2048, N=2048, K=8192) == g.TILE_256x256x64_PAIR    # one wave, long K
    # at most 76 tiles of 128 x 128 and K >= 4096: split-K over two CTAs
    assert g.tile_config(g.TILE_AUTO, M=1024, N=1024, K=8192) == g.TILE_128x128x64_SPLITK
    assert g.tile_config(g.TILE_AUTO, M=128, N=8192, K=8192) == g.TILE_128x128x64_SPLITK
    assert g.tile_config(g.TILE_AUTO, M=1024, N=1024, K=2048) == g.TILE_256x256x128_PAIR
    # at most 38 pair tiles, more than 76 of 128 x 128: k halves from K = 10240
    assert g.tile_config(g.TILE_AUTO, M=1536, N=1536, K=10240) == g.TILE_256x256x64_PAIR_STREAMK
    assert g.tile_config(g.TILE_AUTO, M=1536, N=1536, K=8192) == g.TILE_256x256x128_PAIR
    assert g.tile_config(g.TILE_AUTO, M=2048, N=1024, K=16384) == g.TILE_256x256x64_PAIR_STREAMK
    assert g.tile_config(g.TILE_256x256x128_PAIR_ALIGNED, 8, 8, 8) == g.TILE_256x256x128_PAIR_ALIGNED
    assert g.tile_shape(g.TILE_256x256x64_PAIR_STREAMK) == (256, 256, 64)
    assert g.tile_shape(g.TILE_256x256x64_PAIR) == (256, 256, 64)
    assert g.tile_shape(g.TILE_256x256x128_PAIR) == (256, 256, 128)
    assert g.tile_shape(g.TILE_128x256x64) == (128, 256, 64)
    assert g.tile_shape(g.TILE_128x64x32) == (128, 64, 32)
    assert g.tile_shape(g.TILE_128x128x64) == (128, 128, 64)
    assert g.tile_shape(g.TILE_128x128x64_SPLITK) == (128, 128, 64)
    assert g.tile_shape(g.TILE_128x64x64) == (128, 64, 64)
    assert g.tile_shape(g.TILE_64x64x64) == (64, 64, 64)
    assert g.tile_shape(g.TILE_256x256x128_PAIR_ALIGNED) == (256, 256, 128)
    assert g.TILE_COUNT == 11
    for bad in (17, g.TILE_COUNT, -1):
        with pytest.raises(g.GemmError) as e:
            g.tile_shape(bad)
        assert e.value.code == g.GEMM_ERR_UNSUPPORTED
        with pytest.raises(g.GemmError) as e:
            g.tile_config(bad, 64, 64, 64)
        assert e.value.code == g.GEMM_ERR_UNSUPPORTED
    # every named configuration resolves to itself; AUTO to one of them
    for cfg in range(1, g.TILE_COUNT):
        assert g.tile_config(cfg, 4095, 3000, 1000) == cfg
    assert 1 <= g.tile_config(g.TILE_AUTO, 4095, 3000, 1000) < g.TILE_COUNT


def _call(lib, A=16, B=16, C=16, M=64, N=64, K=64, G=8, cfg=0):
    return lib.gemm_f16_f32acc_tiled(A, B, C, M, N, K, G, cfg, None, None)


def test_aligned_configuration_refuses_partial_tiles_before_any_cuda_call(lib):
    # validation and the whole-tile promise are checked on the host, before a device is touched
    big = 1 << 40
    aligned = g.TILE_256x256x128_PAIR_ALIGNED
    for (M, N, K) in ((255, 256, 128), (256, 264, 128), (256, 256, 136), (4095, 3000, 1000)):
        assert _call(lib, big, 2 * big, 3 * big, M, N, K, cfg=aligned) == g.GEMM_ERR_UNSUPPORTED


def test_validation_without_gpu(lib):
    inv, uns = g.GEMM_ERR_INVALID_ARG, g.GEMM_ERR_UNSUPPORTED
    big = 1 << 40
    assert _call(lib, M=-1) == inv
    assert _call(lib, N=-1) == inv
    assert _call(lib, K=-1) == inv
    assert _call(lib, G=0) == inv
    assert _call(lib, G=-3) == inv
    assert _call(lib, C=0) == inv                       # NULL C with work to do
    assert _call(lib, A=0) == inv                       # NULL A with K > 0
    assert _call(lib, A=25) == uns                      # fp16 needs 2-byte aligned bases
    assert _call(lib, B=big + 1) == uns
    assert _call(lib, C=big + 3) == uns
    assert _call(lib, M=(1 << 30) + 1) == uns
    assert _call(lib, cfg=99) == uns
    # C overlapping A or B
    assert _call(lib, A=big, B=2 * big, C=big + 4096) == inv
    assert _call(lib, A=big, B=2 * big, C=2 * big - 16) == inv
    # no work: OK without touching the device, NULL pointers allowed
    assert _call(lib, A=0, B=0, C=0, M=0) == g.GEMM_OK
    assert _call(lib, A=0, B=0, C=0, N=0) == g.GEMM_OK
    assert lib.gemm_f16_f32acc(0, 0, 0, 0, 5, 5, 1, None) == g.GEMM_OK


def test_tile_schedule_validation_without_gpu(lib):
    assert lib.gemm_tile_schedule(-1, 4, 128, 64, 2, None, None, None) == g.GEMM_ERR_INVALID_ARG
    assert lib.gemm_tile_schedule(4, 4, 0, 64, 2, None, None, None) == g.GEMM_ERR_INVALID_ARG
    assert lib.gemm_tile_schedule(4, 4, 128, 64, 0, None, None, None) == g.GEMM_ERR_INVALID_ARG
    assert lib.gemm_tile_schedule(0, 4, 128, 64, 2, None, None, None) == g.GEMM_OK
    assert lib.gemm_tile_schedule(4, 4, 128, 64, 2, None, None, None) == g.GEMM_ERR_INVALID_ARG


def test_fault_injection_and_watchdog_setters(lib):
    assert lib.gemm_set_fault_injection(2) == g.GEMM_ERR_INVALID_ARG
    assert lib.gemm_set_fault_injection(0) == g.GEMM_OK
    assert lib.gemm_set_watchdog_ns(0) == g.GEMM_OK


def test_python_binding_rejects_host_tensors(lib):
    a = torch.zeros((8, 8), dtype=torch.float16)
    with pytest.raises(ValueError):
        g.gemm(a, a)
    with pytest.raises(TypeError):
        g.gemm(a.float(), a)


def _strided(lib, A=16, lda=64, B=16, ldb=64, C=16, ldc=64, M=64, N=64, K=64):
    return lib.gemm_f16_f32acc_strided(A, lda, B, ldb, C, ldc, M, N, K, 8, 0, None, None)


def test_strided_validation_without_gpu(lib):
    inv, uns = g.GEMM_ERR_INVALID_ARG, g.GEMM_ERR_UNSUPPORTED
    big = 1 << 40
    assert _strided(lib, lda=56) == inv            # pitch shorter than the row
    assert _strided(lib, ldb=63) == inv
    assert _strided(lib, ldc=8) == inv
    assert _strided(lib, ldb=(1 << 30) + 8) == uns
    assert _strided(lib, A=big, lda=1024, B=2 * big, C=big + 1024 * 2 * 63, ldc=1024) == inv  # C inside A's rows
    assert _strided(lib, M=0, A=0, B=0, C=0) == g.GEMM_OK
    assert _strided(lib, A=big + 1, lda=67) == uns     # odd base: not an fp16 address
    # the no-alloc entry point keeps the tensor-map rules (16-byte bases, pitches of 8 elements)
    assert lib.gemm_f16_f32acc_noalloc(16, big, 2 * big, 64, 60, 64, 8, None, None) == uns
    assert lib.gemm_f16_f32acc_noalloc(18, big, 2 * big, 64, 64, 64, 8, None, None) == uns


def test_python_binding_accepts_padded_rows_only(lib):
    base = torch.zeros((8, 16), dtype=torch.float16)
    assert g._binding._row_major(base[:, :10])            # padded rows
    assert not g._binding._row_major(base.t())            # column-major
    assert not g._binding._row_major(base[:, ::2])        # column stride 2
    assert g._binding._ld(base[:, :10]) == 16
    assert g._binding._ld(base[:1, :3]) == 8 and g._binding._ld(torch.zeros((1, 13), dtype=torch.float16)) == 16


def _softmax(lib, X=16, ldx=64, Y=1 << 40, ldy=64, M=8, n=64):
    return lib.softmax_rows_f32(X, ldx, Y, ldy, M, n, None)


def test_softmax_validation_without_gpu(lib):
    inv, uns = g.GEMM_ERR_INVALID_ARG, g.GEMM_ERR_UNSUPPORTED
    big = 1 << 40
    assert _softmax(lib, M=-1) == inv
    assert _softmax(lib, n=-1) == inv
    assert _softmax(lib, ldx=63) == inv                  # pitch shorter than the row
    assert _softmax(lib, ldy=10) == inv
    assert _softmax(lib, X=0) == inv
    assert _softmax(lib, Y=0) == inv
    assert _softmax(lib, n=65537, ldx=70000, ldy=70000) == uns
    assert _softmax(lib, ldx=(1 << 31) + 4) == uns
    assert _softmax(lib, X=18) == uns                    # not 4-byte aligned
    assert _softmax(lib, Y=big + 2) == uns
    # overlapping ranges other than exact in-place
    assert _softmax(lib, X=big, Y=big + 4 * 64 * 7) == inv
    assert _softmax(lib, X=big, Y=big, ldx=64, ldy=128) == inv
    # no work: OK, NULL pointers allowed
    assert _softmax(lib, X=0, Y=0, M=0) == g.GEMM_OK
    assert _softmax(lib, X=0, Y=0, n=0) == g.GEMM_OK


def test_softmax_plan_shapes_without_gpu(lib):
    tpr, cl = ctypes.c_int32(), ctypes.c_int32()
    want = {1: (32, 1), 128: (32, 1), 1024: (32, 1), 1025: (64, 1), 4096: (128, 1), 8192: (256, 1),
            8193: (256, 2), 16384: (256, 2), 16385: (256, 4), 32768: (256, 4), 32769: (256, 8), 65536: (256, 8)}
    for n, shape in want.items():
        assert lib.softmax_rows_plan(10, n, ctypes.byref(tpr), ctypes.byref(cl), None) == g.GEMM_OK
        assert (tpr.value, cl.value) == shape, n
    assert lib.softmax_rows_plan(10, 0, None, None, None) == g.GEMM_ERR_INVALID_ARG
    assert lib.softmax_rows_plan(-1, 8, None, None, None) == g.GEMM_ERR_INVALID_ARG
    assert lib.softmax_rows_plan(10, 65537, None, None, None) == g.GEMM_ERR_UNSUPPORTED


def test_python_softmax_rejects_bad_tensors(lib):
    with pytest.raises(ValueError):
        g.softmax(torch.zeros((4, 8)))                   # host tensor
    with pytest.raises(TypeError):
        g.softmax(torch.zeros((4, 8), dtype=torch.float16))
    assert g._binding._row_pitch(torch.zeros((1, 5))) == 8
    assert g._binding._row_pitch(torch.zeros((3, 16))[:, :5]) == 16


def test_workspace_bytes_without_gpu(lib):
    big = 1 << 40
    need = ctypes.c_uint64(7)
    # every operand suits the tensor maps: no workspace
    assert lib.gemm_workspace_bytes(big, 64, 2 * big, 64, 3 * big, 64, 64, 64, 64, ctypes.byref(need)) == g.GEMM_OK
    assert need.value == 0
    # A pitch 1001 -> copy with pitch 1008; B and C fine
    assert lib.gemm_workspace_bytes(big, 1001, 2 * big, 64, 3 * big, 64, 300, 64, 1001, ctypes.byref(need)) == 0
    assert need.value == -(-(300 * 1008 * 2) // 256) * 256
    # all three: A 300x1008, B 1001x1000, C 300x1000, each region 256-byte aligned
    assert lib.gemm_workspace_bytes(big + 2, 1001, 2 * big, 999, 3 * big + 6, 999, 300, 999, 1001,
                                    ctypes.byref(need)) == 0
    r = lambda x: -(-x // 256) * 256  # noqa: E731
    assert need.value == r(300 * 1008 * 2) + r(1001 * 1000 * 2) + r(300 * 1000 * 2)
    # K == 0: A and B are not read, only C may need a copy
    assert lib.gemm_workspace_bytes(0, 0, 0, 64, 3 * big + 2, 64, 10, 64, 0, ctypes.byref(need)) == 0
    assert need.value == r(10 * 64 * 2)
    # validation as for the GEMM
    assert lib.gemm_workspace_bytes(big, 10, 2 * big, 64, 3 * big, 64, 64, 64, 64,
                                    ctypes.byref(need)) == g.GEMM_ERR_INVALID_ARG
    assert lib.gemm_workspace_bytes(big, 64, 2 * big, 64, 3 * big, 64, 64, 64, 64, None) == g.GEMM_ERR_INVALID_ARG


def test_autotune_validation_without_gpu(lib):
    big = 1 << 40
    args = (big, 64, 2 * big, 64, 3 * big, 64)
    assert lib.gemm_autotune(*args, 64, 64, 64, 8, 0, None, None, None) == g.GEMM_ERR_INVALID_ARG   # reps
    assert lib.gemm_autotune(*args, 64, 64, 64, 8, 10001, None, None, None) == g.GEMM_ERR_INVALID_ARG
    assert lib.gemm_autotune(*args, 0, 64, 64, 8, 5, None, None, None) == g.GEMM_ERR_INVALID_ARG     # nothing to time
    assert lib.gemm_autotune(*args, -1, 64, 64, 8, 5, None, None, None) == g.GEMM_ERR_INVALID_ARG
    assert lib.gemm_autotune(big, 61, 2 * big, 64, 3 * big, 64, 64, 64, 61, 8, 5, None, None,
                             None) == g.GEMM_ERR_UNSUPPORTED                                          # not TMA-shaped
    assert lib.gemm_autotune_clear() == g.GEMM_OK
