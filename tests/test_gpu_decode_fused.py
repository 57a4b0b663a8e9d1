"""GPU parity of the fused and multi-matrix decode entry points.

zq_rmsnorm_q4k_gemv normalises and packs the token inside the mat-vec kernel;
its Q8_1 bytes must equal the oracle's and every output must equal the
two-step path (zq_rmsnorm_q8_1, then zq_q4k_gemv per matrix) bit for bit.
zq_q4k_gemv_multi must equal zq_q4k_gemv per matrix bit for bit.  One shape
per group is also checked against the oracle within 1e-4 * S.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import gemm_zq_rmsnorm_gb300 as zq
from gemm_zq_rmsnorm_gb300 import inputs

from _cases import assert_within, oracle_q8, sample_rows

pytestmark = pytest.mark.gpu


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda")


# (K, [N...]): tiny, ragged, q/k/v, gate/up, o, down, widest K
JOBS = [(256, [1]), (768, [203, 203]), (1024, [1024, 77, 300, 5]), (5120, [6144, 1024, 1024]),
        (5120, [17408, 17408]), (6144, [5120]), (17408, [5120]), (32768, [64, 130])]


def _weights(seed, K, Ns):
    return [inputs.q4k_weights(seed, N, K, tag_offset=7 * m) for m, N in enumerate(Ns)]


@pytest.mark.parametrize("K,Ns", JOBS)
def test_fused_equals_two_step(K, Ns):
    x = inputs.activations(300 + K, 1, K)
    g = inputs.gamma(300 + K, K)
    Ws = [dev(w) for w in _weights(301 + K, K, Ns)]
    xd, gd = dev(x), dev(g)
    a = zq.rmsnorm_q8_1(xd, gd, inputs.EPS)
    ref = [zq.q4k_gemv(W, N, K, a) for W, N in zip(Ws, Ns)]
    q8 = zq.empty_q8_1(1, K)
    got = zq.rmsnorm_q4k_gemv(xd[0], gd, inputs.EPS, Ws, Ns, q8_out=q8)
    torch.cuda.synchronize()
    oq = oracle_q8(x, g)
    assert np.array_equal(q8.qs.cpu().numpy(), oq[0])
    assert np.array_equal(q8.d.cpu().numpy().view(np.uint16), oq[1])
    assert np.array_equal(q8.s.cpu().numpy().view(np.uint16), oq[2])
    for m, (r, y) in enumerate(zip(ref, got)):
        r, y = r.cpu().numpy(), y.cpu().numpy()
        assert np.array_equal(r.view(np.uint32), y.view(np.uint32)), f"matrix {m}: {np.argwhere(r != y)[:5]}"


@pytest.mark.parametrize("K,Ns", [(1024, [1024, 77, 300, 5]), (5120, [6144, 1024, 1024])])
def test_fused_against_oracle(K, Ns):
    x = inputs.activations(310 + K, 1, K)
    g = inputs.gamma(310 + K, K)
    Wn = _weights(311 + K, K, Ns)
    got = zq.rmsnorm_q4k_gemv(dev(x)[0], dev(g), inputs.EPS, [dev(w) for w in Wn], Ns)
    torch.cuda.synchronize()
    qs, d, s = oracle_q8(x, g)
    for W, N, y in zip(Wn, Ns, got):
        rows = sample_rows(N, 7)
        y_ref, S = oracle.q4k_matmul(W, N, K, qs, d, s, rows=rows)
        assert_within(y.cpu().numpy()[None, rows], y_ref, S, f"fused K={K} N={N}")


def test_fused_zero_and_eps_cases():
    K, Ns = 512, [64, 33]
    Wn = _weights(320, K, Ns)
    Ws = [dev(w) for w in Wn]
    g = inputs.gamma(320, K)
    for x, eps in ((np.zeros((1, K), np.float32), inputs.EPS), (np.ones((1, K), np.float32), 0.0),
                   (inputs.activations(321, 1, K), 0.5)):
        a = zq.rmsnorm_q8_1(dev(x), dev(g), eps)
        ref = [zq.q4k_gemv(W, N, K, a) for W, N in zip(Ws, Ns)]
        got = zq.rmsnorm_q4k_gemv(dev(x)[0], dev(g), eps, Ws, Ns)
        torch.cuda.synchronize()
        for r, y in zip(ref, got):
            assert np.array_equal(r.cpu().numpy().view(np.uint32), y.cpu().numpy().view(np.uint32)), eps


@pytest.mark.parametrize("K,Ns", [(1024, [1024, 77, 300, 5]), (5120, [6144, 1024, 1024]), (17408, [5120, 100])])
def test_multi_equals_single(K, Ns):
    x = inputs.activations(330 + K, 1, K)
    g = inputs.gamma(330 + K, K)
    Ws = [dev(w) for w in _weights(331 + K, K, Ns)]
    a = zq.rmsnorm_q8_1(dev(x), dev(g), inputs.EPS)
    ref = [zq.q4k_gemv(W, N, K, a) for W, N in zip(Ws, Ns)]
    got = zq.q4k_gemv_multi(Ws, Ns, K, a)
    torch.cuda.synchronize()
    for r, y in zip(ref, got):
        assert np.array_equal(r.cpu().numpy().view(np.uint32), y.cpu().numpy().view(np.uint32))
