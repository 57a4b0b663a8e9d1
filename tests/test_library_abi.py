"""CPU-only checks of the C-ABI library: it builds, loads, exports every symbol
include/zq.h declares, and rejects bad arguments on the host with the documented
status before touching the device.  No kernel is launched here."""
import ctypes
import os
import re

import pytest

import gemm_zq_rmsnorm_gb300 as zq
from gemm_zq_rmsnorm_gb300 import build as zqbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(zq.LIB_PATH):
        zqbuild.build()
    return zq.load()


def header_functions():
    text = open(os.path.join(ROOT, "include", "zq.h")).read()
    return sorted(set(re.findall(r"ZQ_API\s+[\w\s\*]*?\b(zq_\w+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert header_functions() == sorted(zq.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    for name in header_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_version_and_status_strings(lib):
    assert lib.zq_version() == 1
    for st, text in [(0, b"ok"), (-1, b"invalid argument"), (-2, b"unsupported shape"),
                     (-3, b"misaligned pointer"), (-6, b"workspace missing or too small")]:
        assert lib.zq_status_string(st) == text


def test_size_helpers(lib):
    assert lib.zq_q4k_bytes(5120, 17408) == 5120 * 68 * 144
    assert lib.zq_q4k_bytes(10, 300) == 0
    assert lib.zq_q8_1_bytes(2, 1024) == 2 * 1024 + 2 * 2 * 2 * 32


# fake, never-dereferenced device addresses: validation fails before any use
A16 = 0x10000
A8 = 0x10008


def q8(qs=A16, d=A16, s=A16):
    return zq._Q8(qs, d, s)


@pytest.mark.parametrize("args,status", [
    ((None, A16, 1, 1024, 1e-6, q8()), -1),            # null x
    ((A16, A16, 1, 1000, 1e-6, q8()), -2),             # K % 32
    ((A16, A16, 0, 1024, 1e-6, q8()), -2),             # B = 0
    ((A16, A16, 1, 1024, -1.0, q8()), -1),             # negative eps
    ((A8, A16, 1, 1024, 1e-6, q8()), -3),              # misaligned x
    ((A16, A16, 1, 1024, 1e-6, q8(d=A8)), -3),         # misaligned d plane
])
def test_rmsnorm_rejects(lib, args, status):
    assert lib.zq_rmsnorm_q8_1(*args, None) == status
    assert lib.zq_last_error()


@pytest.mark.parametrize("W,N,K,y,status", [
    (None, 10, 1024, A16, -1), (A16, 0, 1024, A16, -2), (A16, 10, 1000, A16, -2),
    (A16, 10, 0, A16, -2), (A8, 10, 1024, A16, -3), (A16, 10, 1024, A8, -3), (A16, 10, 1024, None, -1)])
def test_gemv_rejects(lib, W, N, K, y, status):
    assert lib.zq_q4k_gemv(W, N, K, q8(), y, None) == status


def test_gemm_rejects(lib):
    assert lib.zq_q4k_gemm(A16, 64, 1024, q8(), 0, A16, None, 0, None) == -2
    assert lib.zq_q4k_gemm(A16, 64, 1024, q8(), 70000, A16, None, 0, None) == -2
    need = lib.zq_q4k_gemm_workspace_bytes(64, 1024, 512)
    if need:
        assert lib.zq_q4k_gemm(A16, 64, 1024, q8(), 512, A16, None, 0, None) == -6
        assert lib.zq_q4k_gemm(A16, 64, 1024, q8(), 512, A16, A16, need - 1, None) == -6
    assert lib.zq_q4k_gemv_pair(A16, None, 64, 1024, q8(), A16, A16, None) == -1
    assert lib.zq_debug_q4k_isums(A16, 64, 1024, q8(), 4, A16, 7, None, 0, None) == -1
    assert lib.zq_debug_q4k_isums(A16, 64, 1024, q8(), 4, A16, 1, None, 0, None) == -2


def test_valid_call_without_gpu_reports_device_error(lib):
    try:
        import torch
        if torch.cuda.is_available():
            pytest.skip("a GPU is present")
    except ImportError:
        pass
    st = lib.zq_q4k_gemv(A16, 64, 1024, q8(), A16, None)
    assert st == -5, lib.zq_last_error()


def test_binding_raises_without_device():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(Exception):
        zq.rmsnorm_q8_1(torch.zeros(1, 64), torch.ones(64), 1e-6)


def _arr(ctype, vals):
    return (ctype * max(len(vals), 1))(*vals)


@pytest.mark.parametrize("nmat,Ws,Ns,ys,K,status", [
    (0, [A16], [10], [A16], 1024, -1),                 # no matrix
    (5, [A16] * 5, [10] * 5, [A16] * 5, 1024, -1),     # more than four
    (2, [A16, None], [10, 10], [A16, A16], 1024, -1),  # null second matrix
    (2, [A16, A16], [10, 0], [A16, A16], 1024, -2),    # N = 0
    (1, [A16], [10], [A16], 1000, -2),                 # K % 256
    (2, [A16, A16], [10, 10], [A16, A8], 1024, -3),    # misaligned y
])
def test_gemv_multi_rejects(lib, nmat, Ws, Ns, ys, K, status):
    W = _arr(ctypes.c_void_p, Ws)
    N = _arr(ctypes.c_int, Ns)
    y = _arr(ctypes.c_void_p, ys)
    assert lib.zq_q4k_gemv_multi(nmat, ctypes.cast(W, ctypes.c_void_p), ctypes.cast(N, ctypes.c_void_p), K, q8(),
                                 ctypes.cast(y, ctypes.c_void_p), None) == status
    assert lib.zq_last_error()


@pytest.mark.parametrize("x,eps,K,nmat,status", [
    (None, 1e-6, 1024, 1, -1),      # null x
    (A8, 1e-6, 1024, 1, -3),        # misaligned x
    (A16, -1.0, 1024, 1, -1),       # negative eps
    (A16, 1e-6, 1024, 0, -1),       # no matrix
    (A16, 1e-6, 33024, 1, -2),      # K above the in-kernel normalisation limit
])
def test_rmsnorm_gemv_rejects(lib, x, eps, K, nmat, status):
    W = _arr(ctypes.c_void_p, [A16])
    N = _arr(ctypes.c_int, [10])
    y = _arr(ctypes.c_void_p, [A16])
    assert lib.zq_rmsnorm_q4k_gemv(x, A16, eps, K, nmat, ctypes.cast(W, ctypes.c_void_p),
                                   ctypes.cast(N, ctypes.c_void_p), ctypes.cast(y, ctypes.c_void_p), None,
                                   None, 0, None) == status
    assert lib.zq_last_error()


@pytest.mark.parametrize("g,u,B,K,status", [
    (None, A16, 1, 64, -1), (A8, A16, 1, 64, -3), (A16, A16, 0, 64, -2), (A16, A16, 1, 48, -2)])
def test_silu_mul_rejects(lib, g, u, B, K, status):
    assert lib.zq_silu_mul_q8_1(g, u, B, K, q8(), None) == status
    assert lib.zq_last_error()


def test_kquant_size_helpers(lib):
    assert lib.zq_q5k_bytes(5120, 6144) == 5120 * 24 * 176
    assert lib.zq_q6k_bytes(151936, 1024) == 151936 * 4 * 210
    assert lib.zq_q5k_bytes(3, 100) == 0 and lib.zq_q6k_bytes(0, 256) == 0


@pytest.mark.parametrize("fn", ["zq_q5k_gemm", "zq_q6k_gemm"])
@pytest.mark.parametrize("W,N,K,B,y,status", [
    (0, 8, 512, 1, A16, -1),          # null W
    (A8, 8, 512, 1, A16, -3),         # misaligned W
    (A16, 0, 512, 1, A16, -2),        # N < 1
    (A16, 8, 500, 1, A16, -2),        # K % 256
    (A16, 8, 33024, 1, A16, -2),      # K above 32768
    (A16, 8, 512, 0, A16, -2),        # B < 1
    (A16, 8, 512, 17, A16, -2),       # B > 16
    (A16, 8, 512, 4, 0, -1),          # null y
    (A16, 8, 512, 4, A8, -3),         # misaligned y
])
def test_kquant_gemm_rejects(lib, fn, W, N, K, B, y, status):
    assert getattr(lib, fn)(W, N, K, q8(), B, y, None) == status


@pytest.mark.parametrize("x,W,K,status", [
    (0, A16, 1024, -1), (A8, A16, 1024, -3), (A16, A8, 1024, -3), (A16, A16, 1000, -2),
    (A16, A16, 33024, -2)])
def test_rmsnorm_q6k_gemv_rejects(lib, x, W, K, status):
    assert lib.zq_rmsnorm_q6k_gemv(x, A16, 1e-6, K, W, 64, A16, None, None) == status


def test_chunk_workspace_query(lib):
    """B = 2..4 run on the streamed mat-vec and need no workspace; from B = 5
    the tensor-core path needs the split activations."""
    for B in (1, 2, 3, 4):
        assert lib.zq_q4k_gemm_workspace_bytes(64, 1024, B) == 0
    assert lib.zq_q4k_gemm_workspace_bytes(64, 1024, 5) >= 4 * 5 * 1024 + 4 * 5
    assert lib.zq_q4k_gemm_workspace_bytes(64, 33024, 4) > 0      # K above the staging limit
    # no workspace needed at B = 4: validation passes, the missing device is reported
    assert lib.zq_q4k_gemm(A16, 64, 1024, q8(), 4, A16, None, 0, None) == -5
    assert lib.zq_q4k_gemm(A16, 64, 1024, q8(), 5, A16, None, 0, None) == -6
    # the integer-sum hook's tensor-core paths need 2*B*K bytes
    assert lib.zq_debug_q4k_isums(A16, 64, 1024, q8(), 4, A16, 2, A16, 2 * 4 * 1024 - 1, None) == -6
    assert lib.zq_debug_q4k_isums(A16, 64, 1024, q8(), 4, A16, 2, A16, 2 * 4 * 1024, None) == -5


def _gemm_base_bytes(B, K):
    """Workspace without partial sums: the binary16 hi and lo halves, the
    token scales and the scaled block sums s8 written twice per super-block
    ([B][K/16] binary16, the min-term operand of both tensor-core kernels);
    each region padded to 256 bytes."""
    pad = lambda n: (n + 255) // 256 * 256
    return 2 * (2 * B * K) + pad(4 * B) + pad(B * (K // 16) * 2)


@pytest.mark.parametrize("K,N", [(5120, 6144), (5120, 1024), (6144, 5120), (5120, 17408), (17408, 5120), (1024, 151936),
                                 (1280, 77), (1280, 65)])
@pytest.mark.parametrize("B", [5, 16, 17, 512])
def test_gemm_workspace_split_k(lib, K, N, B):
    """The workspace holds the binary16 hi and lo activation parts, the token
    scales, the s8 operand and the partial sums.  B >= 17 (2-SM kernel): when
    the launch splits K into S ranges, S partial sums of y, each padded to a
    multiple of four floats (16-byte aligned splits even when B*N is not a
    multiple of 4); S is at most 8 and leaves at least two super-blocks per
    range.  B <= 16 (chunk kernel, contiguous ranges of super-blocks per CTA
    pair): one [B][N] slot per piece of the tile split into the most pieces,
    which is 0 or at least 2 and at most the 256-row tile's super-blocks."""
    ws = lib.zq_q4k_gemm_workspace_bytes(N, K, B)
    base = _gemm_base_bytes(B, K)
    assert ws >= base
    extra = ws - base
    if B <= 16:
        assert extra % (4 * B * N) == 0
        pieces = extra // (4 * B * N)
        assert pieces == 0 or 2 <= pieces <= K // 256 + 1
        return
    stride = 4 * ((B * N + 3) // 4 * 4)
    assert extra % stride == 0
    S = extra // stride
    assert S == 0 or 2 <= S <= 8
    assert S == 0 or (K // 256) // S >= 2


def test_ragged_split_k_shapes_do_split(lib):
    """The GPU parity cases for ragged split-K really split: B*N % 4 != 0 and
    S > 1 (with the fallback SM count used when no device is present)."""
    for (B, K, N) in [(17, 1280, 77), (5, 1280, 65)]:
        assert (B * N) % 4 != 0
        assert lib.zq_q4k_gemm_workspace_bytes(N, K, B) > _gemm_base_bytes(B, K)
