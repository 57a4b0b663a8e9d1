"""Shared helpers for the parity tests: seeded inputs, oracle results and the
tolerance check.  Inputs come only from gemm_zq_rmsnorm_gb300.inputs; expected
values come only from the oracle."""
from __future__ import annotations

import numpy as np

import oracle
from gemm_zq_rmsnorm_gb300 import inputs

# |y_gpu - y_oracle| <= REL_TOL * S, S = sum_k |w_nk * xq_tk| (fp64)
REL_TOL = 1e-4


def sample_rows(N: int, stride: int = 61) -> np.ndarray:
    rows = list(range(0, N, stride))
    if rows[-1] != N - 1:
        rows.append(N - 1)
    return np.asarray(rows, np.int32)


def make_layer_inputs(seed: int, B: int, K: int, N: int, *, tag_offset: int = 0):
    x = inputs.activations(seed, B, K)
    g = inputs.gamma(seed, K)
    W = inputs.q4k_weights(seed, N, K, tag_offset=tag_offset)
    return x, g, W


def assert_within(y_gpu: np.ndarray, y_ref: np.ndarray, S: np.ndarray, what: str):
    y_gpu = np.asarray(y_gpu, np.float64)
    err = np.abs(y_gpu - y_ref.astype(np.float64))
    bound = REL_TOL * S
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5]
        detail = ", ".join(f"{tuple(i)}: gpu={y_gpu[tuple(i)]:.8g} ref={y_ref[tuple(i)]:.8g} "
                           f"err={err[tuple(i)]:.3g} bound={bound[tuple(i)]:.3g}" for i in idx)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside 1e-4*S; {detail}")
    return float((err / np.maximum(S, 1e-300)).max()) if S.size else 0.0


def oracle_q8(x, g, eps=inputs.EPS):
    return oracle.rmsnorm_q8_1(x, g, eps)
