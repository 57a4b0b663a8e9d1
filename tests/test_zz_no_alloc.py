"""The entry point for callers that cannot allocate (zq_q4k_gemm_noalloc).

Some callers of the batched projection have no device memory to hand it:
engines that carve every byte of device memory out of one arena at start-up
and allow no allocation afterwards, and plugins run by a host framework that
gives them no allocator.  zq_q4k_gemm_noalloc serves them from a fixed device
array inside the library.  This test calls it through the C ABI twice in a
row for every batch-size branch that uses the array (B = 5..16: the
small-batch tensor-core kernel; B >= 17: the 128-token tiles) and for B = 4
(the streamed kernel, which needs no scratch), and checks each result against
the oracle (|err| <= 1e-4 * S per element) and against zq_q4k_gemm (which
takes a workspace) within the same tolerance; oversized shapes are refused on
the host.  It sits in a file collected last so that a failure here stops a
`-x` run only after every other test has run; it also passes when run alone
in a fresh process.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import gemm_zq_rmsnorm_gb300 as zq
from gemm_zq_rmsnorm_gb300 import inputs

from _cases import REL_TOL, make_layer_inputs, oracle_q8

pytestmark = pytest.mark.gpu


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda")


def _call_noalloc(lib, W, N, K, a, B, y):
    st = lib.zq_q4k_gemm_noalloc(ctypes.c_void_p(W.data_ptr()), N, K, a._c(), B,
                                 ctypes.c_void_p(y.data_ptr()),
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, lib.zq_last_error().decode()


@pytest.mark.parametrize("B,K,N", [(4, 1024, 300), (8, 1280, 130), (16, 5120, 96), (130, 768, 200),
                                   (512, 5120, 640)])
def test_noalloc_matches_oracle_and_workspace_entry_point(B, K, N):
    lib = zq.load()
    x, g, W = make_layer_inputs(90 + B, B, K, N)
    qs, d, s = oracle_q8(x, g)
    a = zq.Q8_1(_dev(qs), _dev(d.view(np.float16)), _dev(s.view(np.float16)))
    Wd = _dev(W)
    ref = zq.q4k_gemm(Wd, N, K, a, B)          # caller-supplied workspace
    torch.cuda.synchronize()
    ref = ref.cpu().numpy().astype(np.float64)
    # the oracle on every row (a row sample for the 512-token shape)
    rows = np.arange(N, dtype=np.int32) if B * N <= 40000 else np.arange(0, N, 7, dtype=np.int32)
    y_or, S = oracle.q4k_matmul(W, N, K, qs, d, s, rows=rows)
    for call in range(2):                       # two calls in a row share the array
        y = torch.full((B, N), float("nan"), dtype=torch.float32, device="cuda")
        _call_noalloc(lib, Wd, N, K, a, B, y)
        torch.cuda.synchronize()
        got = y.cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(got)), f"call {call}: unwritten outputs"
        err = np.abs(got[:, rows] - y_or)
        assert np.all(err <= REL_TOL * S), f"call {call}: max err/S {np.max(err / np.maximum(S, 1e-300)):.3g}"
        assert np.all(np.abs(got[:, rows] - ref[:, rows]) <= REL_TOL * S), f"call {call} vs zq_q4k_gemm"
        assert np.allclose(got, ref, rtol=0, atol=REL_TOL * float(S.max())), f"call {call}"


def test_noalloc_rejects_oversized_shape_without_launch():
    lib = zq.load()
    B, K, N = 1024, 16384, 256                  # B*K = 16 Mi > 10 Mi
    qs = torch.zeros((B, K), dtype=torch.int8, device="cuda")
    d = torch.zeros((B, K // 32), dtype=torch.float16, device="cuda")
    s = torch.zeros((B, K // 32), dtype=torch.float16, device="cuda")
    W = torch.zeros(zq.q4k_bytes(N, K), dtype=torch.uint8, device="cuda")
    y = torch.zeros((B, N), dtype=torch.float32, device="cuda")
    a = zq.Q8_1(qs, d, s)
    st = lib.zq_q4k_gemm_noalloc(ctypes.c_void_p(W.data_ptr()), N, K, a._c(), B,
                                 ctypes.c_void_p(y.data_ptr()), None)
    assert st == -6, lib.zq_last_error()
