"""GPU parity of SiLU(gate) * up packed to Q8_1 (zq_silu_mul_q8_1) and of the
down-projection launch that computes it inside the mat-vec
(zq_silu_q4k_gemv).  Codes are compared with the oracle bit for bit: both
sides take every step in the library's fp32 definition (exp32, silu, the
Q8_1 packing); the fused launch must equal the two-step path bit for bit."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import gemm_zq_rmsnorm_gb300 as zq
from gemm_zq_rmsnorm_gb300 import inputs

from _cases import assert_within, sample_rows

pytestmark = pytest.mark.gpu


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda")


def gate_up(seed, B, K):
    g = inputs.activations(seed, B, K) * np.float32(1.5)
    u = inputs.activations(seed + 1, B, K)
    # exercise the clamps and the saturating ends of the logistic
    g.flat[:8] = np.array([0.0, -0.0, 86.0, -86.0, 88.0, -88.0, 100.0, -100.0], np.float32)
    return g, u


@pytest.mark.parametrize("B,K", [(1, 64), (1, 17408), (3, 1024), (16, 5120), (512, 3072)])
def test_silu_mul_q8_1_bit_exact(B, K):
    g, u = gate_up(500 + K, B, K)
    a = zq.silu_mul_q8_1(dev(g), dev(u))
    torch.cuda.synchronize()
    qs, d, s = oracle.silu_mul_q8_1(g, u)
    assert np.array_equal(a.qs.cpu().numpy(), qs)
    assert np.array_equal(a.d.cpu().numpy().view(np.uint16), d)
    assert np.array_equal(a.s.cpu().numpy().view(np.uint16), s)


@pytest.mark.parametrize("K,Ns", [(256, [5]), (3072, [1024]), (17408, [5120]), (17408, [5120, 77])])
def test_silu_gemv_fused_equals_two_step(K, Ns):
    g, u = gate_up(510 + K, 1, K)
    Wn = [inputs.q4k_weights(511 + K, N, K, tag_offset=3 * m) for m, N in enumerate(Ns)]
    Ws = [dev(w) for w in Wn]
    a = zq.silu_mul_q8_1(dev(g), dev(u))
    ref = [zq.q4k_gemv(W, N, K, a) for W, N in zip(Ws, Ns)]
    q8 = zq.empty_q8_1(1, K)
    got = zq.silu_q4k_gemv(dev(g)[0], dev(u)[0], Ws, Ns, q8_out=q8)
    torch.cuda.synchronize()
    qs, d, s = oracle.silu_mul_q8_1(g, u)
    assert np.array_equal(q8.qs.cpu().numpy(), qs)
    assert np.array_equal(q8.d.cpu().numpy().view(np.uint16), d)
    for r, y in zip(ref, got):
        assert np.array_equal(r.cpu().numpy().view(np.uint32), y.cpu().numpy().view(np.uint32))
    for W, N, y in zip(Wn, Ns, got):
        rows = sample_rows(N, 13)
        y_ref, S = oracle.q4k_matmul(W, N, K, qs, d, s, rows=rows)
        assert_within(y.cpu().numpy()[None, rows], y_ref, S, f"silu gemv K={K} N={N}")
