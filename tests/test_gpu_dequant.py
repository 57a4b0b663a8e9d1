"""GPU parity of the binary16 dequantisation (zq_q4k_dequant_f16) against the
oracle, bit for bit: both sides take the rounding decisions in the same fp32
steps (a = d*sc, b = dmin*m, a*q - b) and round to binary16."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import gemm_zq_rmsnorm_gb300 as zq
from gemm_zq_rmsnorm_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("N,K", [(1, 256), (77, 768), (300, 5120), (64, 17408)])
def test_dequant_f16_bit_exact(N, K):
    W = inputs.q4k_weights(40 + N, N, K)
    got = zq.q4k_dequant_f16(torch.from_numpy(W).cuda(), N, K)
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy().view(np.uint16), oracle.q4k_dequant_f16(W, N, K))


def test_dequant_f16_extreme_fields():
    N, K = 8, 512
    f = inputs.q4k_fields(41, N, K)
    f.sc[:] = 63
    f.m[:] = 63
    f.q[::2] = 15
    f.q[1::2] = 0
    W = inputs.pack_q4k(f)
    got = zq.q4k_dequant_f16(torch.from_numpy(W).cuda(), N, K)
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy().view(np.uint16), oracle.q4k_dequant_f16(W, N, K))
