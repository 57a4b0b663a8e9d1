"""zq_rmsnorm_q4k_gemm: RMSNorm + Q8_1 and the batched projection in one call.

For B >= 5 the normalisation kernel also writes the binary16 activation
parts, scales and s8 operand that the tensor-core kernels read; the result
must equal zq_rmsnorm_q8_1 followed by zq_q4k_gemm bit for bit, the codes it
returns must equal the oracle's byte for byte, and y must be within the
tolerance of the oracle's projection.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import gemm_zq_rmsnorm_gb300 as zq
from gemm_zq_rmsnorm_gb300 import inputs

from _cases import assert_within, make_layer_inputs, oracle_q8, sample_rows

pytestmark = pytest.mark.gpu

DEV = "cuda"


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


# rows of one block per thread and of two, three and four (K = 8448 leaves
# all but eight threads with one block; K = 32768 is the widest row allowed)
@pytest.mark.parametrize("B,K,N", [(1, 1280, 333), (2, 1280, 333), (4, 2048, 512), (5, 1280, 333),
                                   (16, 5120, 700), (17, 1280, 77), (130, 768, 300), (512, 1024, 512),
                                   (5, 8448, 96), (8, 17408, 64), (6, 32768, 40), (40, 17408, 130)])
def test_fused_equals_two_step(B, K, N):
    x, g, W = make_layer_inputs(300 + B, B, K, N)
    xd, gd, Wd = to_dev(x), to_dev(g), to_dev(W)
    a = zq.rmsnorm_q8_1(xd, gd, inputs.EPS)
    y2 = zq.q4k_gemm(Wd, N, K, a, B)
    q8 = zq.empty_q8_1(B, K, DEV)
    y1 = zq.rmsnorm_q4k_gemm(xd, gd, inputs.EPS, Wd, N, q8_out=q8)
    torch.cuda.synchronize()
    assert zq.device_status() == 0
    assert torch.equal(y1, y2), f"max diff {(y1 - y2).abs().max().item()}"
    qs, d, s = oracle_q8(x, g)
    assert np.array_equal(q8.qs.cpu().numpy(), qs)
    assert np.array_equal(q8.d.cpu().numpy().view(np.uint16), d)
    assert np.array_equal(q8.s.cpu().numpy().view(np.uint16), s)


@pytest.mark.parametrize("K,N", [(5120, 1024), (17408, 256)])
def test_fused_without_codes_and_oracle_prefill(K, N):
    """B = 512 at the attention and down-projection input widths: no q8_out,
    y against the oracle on sampled rows."""
    B = 512
    x, g, W = make_layer_inputs(310, B, K, N)
    y = zq.rmsnorm_q4k_gemm(to_dev(x), to_dev(g), inputs.EPS, to_dev(W), N)
    torch.cuda.synchronize()
    assert zq.device_status() == 0
    qs, d, s = oracle_q8(x, g)
    rows = sample_rows(N, 37)
    y_ref, S = oracle.q4k_matmul(W, N, K, qs, d, s, rows=rows)
    assert_within(y.cpu().numpy()[:, rows], y_ref, S, f"rmsnorm_q4k_gemm B=512 K={K}")


def test_fused_argument_checks():
    K, N, B = 256, 8, 3
    x = torch.zeros((B, K), dtype=torch.float32, device=DEV)
    g = torch.ones(K, dtype=torch.float32, device=DEV)
    W = torch.zeros(zq.q4k_bytes(N, K), dtype=torch.uint8, device=DEV)
    y = torch.empty((B, N), dtype=torch.float32, device=DEV)
    lib = zq.load()
    # B = 3 runs the streamed mat-vec, which reads the codes: q8_out is required
    st = lib.zq_rmsnorm_q4k_gemm(x.data_ptr(), g.data_ptr(), 1e-6, B, K, W.data_ptr(), N, y.data_ptr(), None,
                                 None, 0, None)
    assert st == -1   # ZQ_ERR_ARG
    # K above the in-kernel normalisation limit
    K2 = 33024
    with pytest.raises(zq.ZQError):
        zq.rmsnorm_q4k_gemm(torch.zeros((6, K2), dtype=torch.float32, device=DEV), torch.ones(K2, device=DEV),
                            1e-6, torch.zeros(zq.q4k_bytes(8, K2), dtype=torch.uint8, device=DEV), 8)
