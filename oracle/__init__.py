"""CPU oracle of the quantized projection (test infrastructure only).

Only the test-suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never does, and
the oracle imports nothing from the product package: the two sides share only
the seeded input generators of ``gemm_zq_rmsnorm_gb300.inputs``.

The arithmetic lives in ``zq_oracle.c`` (plain single-threaded C, compiled with
floating-point contraction off).  This module builds it with the host C
compiler and exposes numpy wrappers with the same names.

Every function is pinned by ``tests/test_oracle_pins.py`` against hand-worked
examples, closed forms, library routines and brute force; none of it is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "zq_oracle.c")
_LIB = os.path.join(_HERE, "libzq_oracle.so")
_CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC"]

_lib = None


def build(force: bool = False) -> str:
    """Compile ``zq_oracle.c`` into ``libzq_oracle.so`` next to it."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cc = os.environ.get("CC", "gcc")
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call([cc, *_CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i, f = ctypes.c_int, ctypes.c_float
        lib.zqo_f32_to_f16.argtypes = [f]
        lib.zqo_f32_to_f16.restype = ctypes.c_uint16
        lib.zqo_f32_to_f16_array.argtypes = [P, P, ctypes.c_size_t]
        lib.zqo_f32_to_f16_array.restype = None
        lib.zqo_f16_to_f32.argtypes = [ctypes.c_uint16]
        lib.zqo_f16_to_f32.restype = f
        lib.zqo_rms_scale.argtypes = [P, i, f]
        lib.zqo_rms_scale.restype = f
        lib.zqo_rmsnorm_q8_1.argtypes = [P, P, i, i, f, P, P, P]
        lib.zqo_rmsnorm_q8_1.restype = None
        lib.zqo_q4k_unpack.argtypes = [P, P, P, P, P, P]
        lib.zqo_q4k_unpack.restype = None
        lib.zqo_q4k_dequant.argtypes = [P, i, i, P]
        lib.zqo_q4k_dequant.restype = None
        lib.zqo_q4k_dequant_f16.argtypes = [P, i, i, P]
        lib.zqo_q4k_dequant_f16.restype = None
        lib.zqo_q8_1_dequant_f16.argtypes = [P, P, i, i, P]
        lib.zqo_q8_1_dequant_f16.restype = None
        lib.zqo_f16_gemm_rows.argtypes = [P, P, i, i, P, i, P]
        lib.zqo_f16_gemm_rows.restype = None
        lib.zqo_exp32.argtypes = [f]
        lib.zqo_exp32.restype = f
        lib.zqo_silu32.argtypes = [f]
        lib.zqo_silu32.restype = f
        lib.zqo_silu_mul_q8_1.argtypes = [P, P, i, i, P, P, P]
        lib.zqo_silu_mul_q8_1.restype = None
        lib.zqo_q4k_isums.argtypes = [P, i, i, P, i, P]
        lib.zqo_q4k_isums.restype = None
        lib.zqo_q4k_matmul_rows.argtypes = [P, i, i, P, P, P, i, P, i, P, P]
        lib.zqo_q4k_matmul_rows.restype = None
        lib.zqo_q5k_unpack.argtypes = [P, P, P, P, P, P]
        lib.zqo_q5k_unpack.restype = None
        lib.zqo_q6k_unpack.argtypes = [P, P, P, P]
        lib.zqo_q6k_unpack.restype = None
        lib.zqo_q5k_dequant.argtypes = [P, i, i, P]
        lib.zqo_q5k_dequant.restype = None
        lib.zqo_q6k_dequant.argtypes = [P, i, i, P]
        lib.zqo_q6k_dequant.restype = None
        lib.zqo_q5k_matmul_rows.argtypes = [P, i, i, P, P, P, i, P, i, P, P]
        lib.zqo_q5k_matmul_rows.restype = None
        lib.zqo_q6k_matmul_rows.argtypes = [P, i, i, P, P, i, P, i, P, P]
        lib.zqo_q6k_matmul_rows.restype = None
        _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def f32_to_f16_bits(v) -> np.ndarray:
    """Binary16 bit patterns (uint16) of fp32 values, RNE, from the IEEE definition."""
    a = np.ascontiguousarray(np.asarray(v, dtype=np.float32).ravel())
    h = np.zeros(a.size, np.uint16)
    _load().zqo_f32_to_f16_array(_p(a), _p(h), a.size)
    return h


def f16_bits_to_f32(h) -> np.ndarray:
    lib = _load()
    a = np.asarray(h, dtype=np.uint16).ravel()
    return np.array([lib.zqo_f16_to_f32(int(x)) for x in a], dtype=np.float32)


def rms_scale(x: np.ndarray, eps: float) -> np.float32:
    """r = 1/sqrt(ss/K + eps) for one token, in the fixed fp32 order."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    return np.float32(_load().zqo_rms_scale(_p(x), x.shape[-1], eps))


def rmsnorm_q8_1(x: np.ndarray, gamma: np.ndarray, eps: float):
    """Fused RMSNorm + Q8_1 pack.  x fp32 [B][K] -> (qs int8 [B][K],
    d uint16 [B][K/32] (fp16 bits), s uint16 [B][K/32] (fp16 bits))."""
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float32)
    g = np.ascontiguousarray(gamma, dtype=np.float32)
    B, K = x.shape
    assert K % 32 == 0 and g.shape == (K,)
    qs = np.zeros((B, K), np.int8)
    d = np.zeros((B, K // 32), np.uint16)
    s = np.zeros((B, K // 32), np.uint16)
    _load().zqo_rmsnorm_q8_1(_p(x), _p(g), B, K, eps, _p(qs), _p(d), _p(s))
    return qs, d, s


def exp32(a) -> np.ndarray:
    """The library's fp32 exponential (range reduction + degree-7 polynomial)."""
    lib = _load()
    return np.array([lib.zqo_exp32(float(v)) for v in np.asarray(a, np.float32).ravel()], np.float32)


def silu32(g) -> np.ndarray:
    """silu(g) = g / (1 + exp32(-g)), fp32 steps."""
    lib = _load()
    return np.array([lib.zqo_silu32(float(v)) for v in np.asarray(g, np.float32).ravel()], np.float32)


def silu_mul_q8_1(g: np.ndarray, u: np.ndarray):
    """Q8_1 of silu(g) * u (fp32 [B][K] each) -> (qs, d bits, s bits)."""
    g = np.ascontiguousarray(np.atleast_2d(g), dtype=np.float32)
    u = np.ascontiguousarray(np.atleast_2d(u), dtype=np.float32)
    B, K = g.shape
    assert u.shape == g.shape and K % 32 == 0
    qs = np.zeros((B, K), np.int8)
    d = np.zeros((B, K // 32), np.uint16)
    s = np.zeros((B, K // 32), np.uint16)
    _load().zqo_silu_mul_q8_1(_p(g), _p(u), B, K, _p(qs), _p(d), _p(s))
    return qs, d, s


def q4k_unpack(block: np.ndarray):
    """One 144-byte Q4_K super-block -> (d, dmin, sc[8], m[8], q[256])."""
    blk = np.ascontiguousarray(block, dtype=np.uint8)
    assert blk.size == 144
    d = ctypes.c_float()
    dmin = ctypes.c_float()
    sc = np.zeros(8, np.uint8)
    m = np.zeros(8, np.uint8)
    q = np.zeros(256, np.uint8)
    _load().zqo_q4k_unpack(_p(blk), ctypes.byref(d), ctypes.byref(dmin), _p(sc), _p(m), _p(q))
    return np.float32(d.value), np.float32(dmin.value), sc, m, q


def q4k_dequant(W: np.ndarray, N: int, K: int) -> np.ndarray:
    W = np.ascontiguousarray(W, dtype=np.uint8)
    assert W.size == N * (K // 256) * 144
    w = np.zeros((N, K), np.float64)
    _load().zqo_q4k_dequant(_p(W), N, K, _p(w))
    return w


def q4k_dequant_f16(W: np.ndarray, N: int, K: int) -> np.ndarray:
    """Binary16 bit patterns [N][K] of the weights, via fp32 a*q - b (see
    zqo_q4k_dequant_f16)."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    assert W.size == N * (K // 256) * 144
    w = np.zeros((N, K), np.uint16)
    _load().zqo_q4k_dequant_f16(_p(W), N, K, _p(w))
    return w


def q8_1_dequant_f16(qs: np.ndarray, d: np.ndarray) -> np.ndarray:
    """Binary16 bit patterns [B][K] of x = q8 * d8 (see zqo_q8_1_dequant_f16)."""
    qs = np.ascontiguousarray(np.atleast_2d(qs), dtype=np.int8)
    d = np.ascontiguousarray(np.atleast_2d(d), dtype=np.uint16)
    B, K = qs.shape
    assert K % 32 == 0 and d.shape == (B, K // 32)
    x = np.zeros((B, K), np.uint16)
    _load().zqo_q8_1_dequant_f16(_p(qs), _p(d), B, K, _p(x))
    return x


def f16_gemm(x16: np.ndarray, w16: np.ndarray, rows=None) -> np.ndarray:
    """y[t][r] (fp64) = sum_k x16[t][k] * w16[rows[r]][k] of binary16 bit
    patterns x16 [B][K] and w16 [N][K] (see zqo_f16_gemm_rows)."""
    x16 = np.ascontiguousarray(np.atleast_2d(x16), dtype=np.uint16)
    w16 = np.ascontiguousarray(w16, dtype=np.uint16)
    B, K = x16.shape
    N = w16.shape[0]
    assert w16.shape == (N, K)
    r = np.arange(N, dtype=np.int32) if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    y = np.zeros((B, r.size), np.float64)
    _load().zqo_f16_gemm_rows(_p(x16), _p(w16), B, K, _p(r), r.size, _p(y))
    return y


def q4k_isums(W: np.ndarray, N: int, K: int, qs: np.ndarray) -> np.ndarray:
    """I[t][n][K/32] exact int32 sub-block dot sums."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    qs = np.ascontiguousarray(np.atleast_2d(qs), dtype=np.int8)
    B = qs.shape[0]
    I = np.zeros((B, N, K // 32), np.int32)
    _load().zqo_q4k_isums(_p(W), N, K, _p(qs), B, _p(I))
    return I


def q4k_matmul(W, N, K, qs, d, s, rows=None, want_scale=True):
    """y[t][r] (fp32) for rows r (all when None) and the tolerance scale
    S[t][r] = sum_k |w*xq| (fp64) when want_scale."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    qs = np.ascontiguousarray(np.atleast_2d(qs), dtype=np.int8)
    d = np.ascontiguousarray(np.atleast_2d(d), dtype=np.uint16)
    s = np.ascontiguousarray(np.atleast_2d(s), dtype=np.uint16)
    B = qs.shape[0]
    assert qs.shape[1] == K and d.shape == (B, K // 32) and s.shape == (B, K // 32)
    if rows is None:
        R = N
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int32)
        R = rows_arr.size
        assert rows_arr.min() >= 0 and rows_arr.max() < N
    y = np.zeros((B, R), np.float32)
    S = np.zeros((B, R), np.float64) if want_scale else None
    _load().zqo_q4k_matmul_rows(
        _p(W), N, K, _p(qs), _p(d), _p(s), B,
        _p(rows_arr) if rows_arr is not None else None, R, _p(y),
        _p(S) if S is not None else None)
    return (y, S) if want_scale else y


# ---------------------------------------------------------------- Q5_K, Q6_K
BLOCK_BYTES = {"q4k": 144, "q5k": 176, "q6k": 210}


def q5k_unpack(block: np.ndarray):
    """One 176-byte Q5_K super-block -> (d, dmin, sc[8], m[8], q[256] 0..31)."""
    blk = np.ascontiguousarray(block, dtype=np.uint8)
    assert blk.size == 176
    d = ctypes.c_float()
    dmin = ctypes.c_float()
    sc = np.zeros(8, np.uint8)
    m = np.zeros(8, np.uint8)
    q = np.zeros(256, np.uint8)
    _load().zqo_q5k_unpack(_p(blk), ctypes.byref(d), ctypes.byref(dmin), _p(sc), _p(m), _p(q))
    return np.float32(d.value), np.float32(dmin.value), sc, m, q


def q6k_unpack(block: np.ndarray):
    """One 210-byte Q6_K super-block -> (d, sc[16] int8, q[256] 0..63)."""
    blk = np.ascontiguousarray(block, dtype=np.uint8)
    assert blk.size == 210
    d = ctypes.c_float()
    sc = np.zeros(16, np.int8)
    q = np.zeros(256, np.uint8)
    _load().zqo_q6k_unpack(_p(blk), ctypes.byref(d), _p(sc), _p(q))
    return np.float32(d.value), sc, q


def kq_dequant(fmt: str, W: np.ndarray, N: int, K: int) -> np.ndarray:
    """fp64 weights [N][K] of a Q5_K ("q5k") or Q6_K ("q6k") matrix."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    assert W.size == N * (K // 256) * BLOCK_BYTES[fmt]
    w = np.zeros((N, K), np.float64)
    fn = {"q5k": _load().zqo_q5k_dequant, "q6k": _load().zqo_q6k_dequant}[fmt]
    fn(_p(W), N, K, _p(w))
    return w


def kq_matmul(fmt, W, N, K, qs, d, s, rows=None, want_scale=True):
    """q4k_matmul for a matrix of format fmt ("q4k", "q5k" or "q6k")."""
    if fmt == "q4k":
        return q4k_matmul(W, N, K, qs, d, s, rows=rows, want_scale=want_scale)
    W = np.ascontiguousarray(W, dtype=np.uint8)
    assert W.size == N * (K // 256) * BLOCK_BYTES[fmt]
    qs = np.ascontiguousarray(np.atleast_2d(qs), dtype=np.int8)
    d = np.ascontiguousarray(np.atleast_2d(d), dtype=np.uint16)
    s = np.ascontiguousarray(np.atleast_2d(s), dtype=np.uint16)
    B = qs.shape[0]
    assert qs.shape[1] == K and d.shape == (B, K // 32) and s.shape == (B, K // 32)
    if rows is None:
        R, rows_arr = N, None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int32)
        R = rows_arr.size
        assert rows_arr.min() >= 0 and rows_arr.max() < N
    y = np.zeros((B, R), np.float32)
    S = np.zeros((B, R), np.float64) if want_scale else None
    rp = _p(rows_arr) if rows_arr is not None else None
    Sp = _p(S) if S is not None else None
    if fmt == "q5k":
        _load().zqo_q5k_matmul_rows(_p(W), N, K, _p(qs), _p(d), _p(s), B, rp, R, _p(y), Sp)
    else:
        _load().zqo_q6k_matmul_rows(_p(W), N, K, _p(qs), _p(d), B, rp, R, _p(y), Sp)
    return (y, S) if want_scale else y
