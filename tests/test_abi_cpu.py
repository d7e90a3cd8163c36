"""The C ABI on a machine without a GPU: the library builds, loads, exports
every entry point include/q4_0.h declares, and rejects bad arguments before
touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "q4_0.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(q4_0_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from q4_weight_only_gb300 import build, _lib
    build.build()
    return _lib.lib()


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("q4_0_quantize", "q4_0_matmul", "q4_0_status_string", "q4_0_version",
                     "q4_0_weight_bytes"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    from q4_weight_only_gb300 import _lib
    names = declared_functions()
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(_lib.SIGNATURES) == names


def test_version_and_status_strings(lib):
    assert lib.q4_0_version() == 1
    for code in (0, -1, -2, -3, -4, -5, 7):
        assert lib.q4_0_status_string(code)


def test_weight_bytes(lib):
    assert lib.q4_0_weight_bytes(256, 1024) == 256 * 32 * 18
    assert lib.q4_0_weight_bytes(7168, 5120) == 20643840
    assert lib.q4_0_weight_bytes(1, 33) == 0
    assert lib.q4_0_weight_bytes(0, 32) == 0


def test_workspace_sizes(lib):
    a256 = lambda b: (b + 255) // 256 * 256
    # batched decode (no device here, so no room for split-K partials): x as
    # binary16 tiles of 16 or 32 rows, then 256 bytes for the rows' scales
    tc = lambda tm, K: a256(tm * K * 2) + 256
    # GEMM (unsplit): x as binary16, then the rows' scales
    gemm = lambda M, K: a256(M * K * 2) + a256(M * 4)
    assert lib.q4_0_matmul_workspace_bytes(1, 5120, 5120) == 0
    assert lib.q4_0_matmul_workspace_bytes(2, 5120, 5120) == 0
    assert lib.q4_0_matmul_workspace_bytes(3, 5120, 5120) == tc(16, 5120)
    assert lib.q4_0_matmul_workspace_bytes(16, 5120, 17408) == tc(16, 17408)
    assert lib.q4_0_matmul_workspace_bytes(17, 5120, 5120) == tc(32, 5120)
    assert lib.q4_0_matmul_workspace_bytes(32, 5120, 5120) == tc(32, 5120)
    for M in (1, 2, 3, 16, 17, 32, 33, 64):
        assert lib.q4_0_gemv_workspace_bytes(M, 5120) == lib.q4_0_matmul_workspace_bytes(M, 7, 5120)
    assert lib.q4_0_matmul_workspace_bytes(33, 5120, 5120) == tc(64, 5120)
    assert lib.q4_0_matmul_workspace_bytes(64, 5120, 5120) == tc(64, 5120)
    assert lib.q4_0_gemv_workspace_bytes(64, 5120) == tc(64, 5120)
    assert lib.q4_0_gemv_workspace_bytes(65, 5120) == 0
    # K % 256 != 0: zero-padded copies of W and x (256-byte aligned), then the
    # padded problem's own scratch
    assert lib.q4_0_matmul_workspace_bytes(1, 300, 96) == a256(300 * 8 * 18) + a256(1 * 256 * 2)
    assert lib.q4_0_matmul_workspace_bytes(16, 300, 5152) == (a256(300 * 168 * 18) + a256(16 * 5376 * 2)
                                                               + tc(16, 5376))
    assert lib.q4_0_matmul_workspace_bytes(64, 300, 288) >= a256(300 * 16 * 18) + a256(64 * 512 * 2) + gemm(64, 512)
    assert lib.q4_0_matmul_workspace_bytes(65, 5120, 5120) == gemm(65, 5120)
    assert lib.q4_0_gemm_workspace_bytes(3, 128, 256) % 256 == 0
    # one or two rows with K past 65536 (x no longer fits shared memory) take
    # the tensor-core decode and its x tiles
    for M in (1, 2):
        assert lib.q4_0_matmul_workspace_bytes(M, 300, 65536) == 0
        assert lib.q4_0_matmul_workspace_bytes(M, 300, 65792) == tc(16, 65792)
        assert lib.q4_0_gemv_workspace_bytes(M, 131072) == tc(16, 131072)


def test_invalid_arguments_rejected_before_cuda(lib):
    P = ctypes.c_void_p
    good = P(1 << 20)  # never dereferenced: validation fails first
    assert lib.q4_0_matmul(None, good, good, 1, 1, 256, None) == -1
    assert lib.q4_0_matmul(good, good, good, 0, 1, 256, None) == -1
    assert lib.q4_0_matmul(good, good, good, 1, 0, 256, None) == -1
    assert lib.q4_0_matmul(good, good, good, 1, 1, 48, None) == -1     # K % 32
    assert lib.q4_0_gemm(good, good, good, 64, 1, 96, good, 1 << 20, None) == -2   # kernel alone: K % 256
    assert lib.q4_0_gemv_ws(good, good, good, 1, 1, 96, None, 0, None) == -2
    assert lib.q4_0_matmul(P((1 << 20) + 8), good, good, 1, 1, 256, None) == -1  # misaligned
    assert lib.q4_0_gemv(good, good, good, 65, 1, 256, None) == -2
    assert lib.q4_0_matmul_ex(good, good, good, 7, 1, 1, 256, None, 0, None) == -1   # unknown y type
    assert lib.q4_0_matmul_ex(good, good, good, 1, 1, 1, 48, None, 0, None) == -1    # K % 32
    assert lib.q4_0_gemv_ws(good, good, good, 16, 1, 256, None, 0, None) == -5
    assert lib.q4_0_gemv_ws(good, good, good, 16, 1, 256, P((1 << 20) + 16), 1 << 20, None) == -5
    assert lib.q4_0_gemv_ws(good, good, good, 16, 1, 256, good, 16 * 256 * 2 - 1, None) == -5
    assert lib.q4_0_gemm(good, good, good, 64, 1, 256, None, 0, None) == -5
    assert lib.q4_0_gemm(good, good, good, 64, 1, 256, P((1 << 20) + 16), 1 << 20, None) == -5
    assert lib.q4_0_quantize(None, good, 1, 32, None) == -1
    assert lib.q4_0_quantize(good, good, 1, 31, None) == -1
    assert lib.q4_0_device_error(None) == -1


def test_shapes_past_the_grid_limits_are_unsupported(lib):
    """Shapes the launch grids cannot hold are refused before any CUDA call:
    the tensor-core decode's weight tiles (N <= 65535 * 128), and sizes past
    the caps (M, N <= 2^30; the GEMM's one-dimensional grid of tiles then
    always fits)."""
    good = ctypes.c_void_p(1 << 20)
    ws = ctypes.c_void_p(1 << 21)
    assert lib.q4_0_matmul_ws(good, good, good, 16, 65535 * 128 + 1, 256, ws, 1 << 40, None) == -2
    assert lib.q4_0_matmul_ws(good, good, good, 1, 65535 * 128 + 1, 65792, ws, 1 << 40, None) == -2
    assert lib.q4_0_gemv_ws(good, good, good, 16, 65535 * 128 + 1, 256, ws, 1 << 40, None) == -2
    assert lib.q4_0_gemm(good, good, good, (1 << 30) + 1, 128, 256, ws, 1 << 40, None) == -2
    assert lib.q4_0_matmul_ws(good, good, good, (1 << 30) + 1, 128, 256, ws, 1 << 40, None) == -2


def test_grouped_validates_every_problem_before_any_launch(lib):
    """q4_0_matmul_grouped checks the whole group first: a bad count, array,
    output type or problem anywhere in it is refused before any CUDA call."""
    P = ctypes.c_void_p
    G = 3
    ptrs = (P * G)(*([1 << 20] * G))
    ns = (ctypes.c_int64 * G)(5120, 5120, 5120)
    ks = (ctypes.c_int64 * G)(5120, 5120, 5120)
    c = lambda a: ctypes.cast(a, P)
    assert lib.q4_0_matmul_grouped(0, None, None, None, 0, 1, None, None, None) == 0   # nothing to do
    assert lib.q4_0_matmul_grouped(-1, c(ptrs), c(ptrs), c(ptrs), 0, 1, c(ns), c(ks), None) == -1
    assert lib.q4_0_matmul_grouped(G, None, c(ptrs), c(ptrs), 0, 1, c(ns), c(ks), None) == -1
    assert lib.q4_0_matmul_grouped(G, c(ptrs), c(ptrs), c(ptrs), 0, 1, c(ns), None, None) == -1
    assert lib.q4_0_matmul_grouped(G, c(ptrs), c(ptrs), c(ptrs), 7, 1, c(ns), c(ks), None) == -1
    bad_k = (ctypes.c_int64 * G)(5120, 5120, 48)        # the last problem: K % 32 != 0
    assert lib.q4_0_matmul_grouped(G, c(ptrs), c(ptrs), c(ptrs), 0, 1, c(ns), c(bad_k), None) == -1
    misaligned = (P * G)(1 << 20, (1 << 20) + 8, 1 << 20)
    assert lib.q4_0_matmul_grouped(G, c(misaligned), c(ptrs), c(ptrs), 0, 1, c(ns), c(ks), None) == -1
    too_tall = (ctypes.c_int64 * G)(5120, 65535 * 128 + 1, 5120)   # tensor-core decode grid limit
    assert lib.q4_0_matmul_grouped(G, c(ptrs), c(ptrs), c(ptrs), 0, 16, c(too_tall), c(ks), None) == -2


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    from q4_weight_only_gb300 import _lib
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(RuntimeError):
        _lib.lib()


def test_matmul_host_validates_before_any_copy(lib):
    """q4_0_matmul_host rejects bad arguments before touching the GPU."""
    p = ctypes.c_void_p(16)
    # bad output type, null host buffers
    assert lib.q4_0_matmul_host(p, p, p, 7, 1, 128, 256, p, 1 << 20, None) == -1
    assert lib.q4_0_matmul_host(None, p, p, 0, 1, 128, 256, p, 1 << 20, None) == -1
    assert lib.q4_0_matmul_host(p, p, None, 0, 1, 128, 256, p, 1 << 20, None) == -1
    # K not a multiple of 32
    assert lib.q4_0_matmul_host(p, p, p, 0, 1, 128, 100, p, 1 << 20, None) == -1
    # missing, small or misaligned workspace
    need = lib.q4_0_matmul_host_workspace_bytes(4, 128, 256, 0)
    assert lib.q4_0_matmul_host(p, p, p, 0, 4, 128, 256, None, 0, None) == -5
    assert lib.q4_0_matmul_host(p, p, p, 0, 4, 128, 256, p, need - 1, None) == -5
    assert lib.q4_0_matmul_host(p, p, p, 0, 4, 128, 256, ctypes.c_void_p(24), need, None) == -5


def test_matmul_host_workspace_sizes(lib):
    """Device copies of x and y (each rounded up to 256 bytes), then the
    dispatcher's own scratch; 0 for arguments the call rejects."""
    for M, N, K, yt in ((1, 5120, 5120, 0), (16, 300, 2048, 1), (300, 500, 1024, 0), (3, 100, 96, 1)):
        ysz = 2 if yt else 4
        x = (M * K * 2 + 255) // 256 * 256
        y = (M * N * ysz + 255) // 256 * 256
        assert lib.q4_0_matmul_host_workspace_bytes(M, N, K, yt) == x + y + lib.q4_0_matmul_workspace_bytes(M, N, K)
    assert lib.q4_0_matmul_host_workspace_bytes(1, 128, 256, 2) == 0
    assert lib.q4_0_matmul_host_workspace_bytes(0, 128, 256, 0) == 0
    assert lib.q4_0_matmul_host_workspace_bytes(1, 128, 100, 0) == 0


def test_grouped_binding_checks_its_lists(lib):
    """matmul_grouped: an empty group is a no-op and lists of different
    lengths are refused before anything reaches the library."""
    import q4_weight_only_gb300 as q4
    assert q4.matmul_grouped([], [], [], []) == []
    with pytest.raises(ValueError):
        q4.matmul_grouped([None], [None, None], [1], [32])
    with pytest.raises(ValueError):
        q4.matmul_grouped([None], [None], [1], [32], outs=[None, None])
    assert q4.grouped_launches(1, [], []) == -1
