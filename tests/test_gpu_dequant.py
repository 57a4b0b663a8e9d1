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


# ------------------------------------------------ dequantise-then-GEMM (f3)
from _cases import assert_within, make_layer_inputs, oracle_q8, sample_rows  # noqa: E402


def q8_dev(qs, d, s) -> zq.Q8_1:
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    return zq.Q8_1(dev(qs), dev(d.view(np.float16)), dev(s.view(np.float16)))


@pytest.mark.parametrize("B,K", [(1, 256), (5, 1280), (512, 5120), (3, 17408)])
def test_q8_1_dequant_f16_bit_exact(B, K):
    x, g, _ = make_layer_inputs(70 + B, B, K, 1)
    qs, d, s = oracle_q8(x, g)
    got = zq.q8_1_dequant_f16(q8_dev(qs, d, s))
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy().view(np.uint16), oracle.q8_1_dequant_f16(qs, d))


def f16_gemm_case(B, N, K, seed, rows=None):
    """GPU dequantise-then-GEMM on seeded Q4_K weights and Q8_1 activations,
    with the oracle's binary16 operands and its fp64 GEMM of them."""
    x, g, W = make_layer_inputs(seed, B, K, N)
    qs, d, s = oracle_q8(x, g)
    x16 = oracle.q8_1_dequant_f16(qs, d)
    w16 = oracle.q4k_dequant_f16(W, N, K)
    Wd = torch.from_numpy(W).cuda()
    W16 = zq.q4k_dequant_f16(Wd, N, K)
    X16 = zq.q8_1_dequant_f16(q8_dev(qs, d, s))
    y = zq.f16_gemm(W16, N, K, X16, B)
    torch.cuda.synchronize()
    assert zq.device_status() == 0
    y = y.cpu().numpy()
    if rows is None:
        rows = np.arange(N, dtype=np.int32)
    y_ref = oracle.f16_gemm(x16, w16, rows=rows)
    S16 = oracle.f16_gemm(x16 & 0x7FFF, w16 & 0x7FFF, rows=rows)   # sum |x16 * w16|
    return y[:, rows], y_ref, S16, (W, qs, d, s, rows)


@pytest.mark.parametrize("B,N,K", [
    (17, 77, 256),       # ragged tokens and rows, one stage of K
    (5, 1000, 1024),     # a 16-token tile
    (130, 300, 1280),    # two token tiles, ragged
    (256, 512, 5120),    # whole tiles
    (64, 256, 17408),    # one tile: split over K
    (300, 1100, 2048),
])
def test_f16_gemm_all_outputs(B, N, K):
    """Every output of the binary16 GEMM within 1e-4 of sum |x16*w16| of the
    oracle's fp64 GEMM of the same binary16 operands (fp32 accumulation)."""
    y, y_ref, S16, _ = f16_gemm_case(B, N, K, 80 + B)
    assert_within(y, y_ref, S16, f"f16 gemm B={B} N={N} K={K}")


def test_f16_gemm_gate_512_sampled_and_error_vs_q4k():
    """The 512-token gate shape, sampled rows: against the oracle's GEMM of
    the same binary16 operands, and against the Q4_K x Q8_1 projection's
    oracle, where the two binary16 roundings (weights, activations) bound the
    error by about 2^-10 * S."""
    B, N, K = 512, 17408, 5120
    rows = sample_rows(N, 127)
    y, y_ref, S16, (W, qs, d, s, rows) = f16_gemm_case(B, N, K, 90, rows=rows)
    assert_within(y, y_ref, S16, "f16 gemm gate (same operands)")
    yq, S = oracle.q4k_matmul(W, N, K, qs, d, s, rows=rows)
    err = np.abs(y.astype(np.float64) - yq.astype(np.float64))
    ratio = float((err / np.maximum(S, 1e-30)).max())
    print(f"dequantise-then-GEMM vs Q4_K x Q8_1 oracle: max err / S = {ratio:.3e}")
    assert np.all(err <= 1.1e-3 * S + 1e-6), ratio


def test_f16_gemm_workspace_checks():
    N, K, B = 256, 17408, 64
    need = zq.f16_gemm_workspace_bytes(N, K, B)
    assert need > 0   # one tile: the call splits K
    W16 = torch.zeros((N, K), dtype=torch.float16, device="cuda")
    X16 = torch.zeros((B, K), dtype=torch.float16, device="cuda")
    ws = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(zq.ZQError):
        zq.f16_gemm(W16, N, K, X16, B, workspace=ws)
    with pytest.raises(zq.ZQError):
        zq.f16_gemm(W16, N, 100, X16, B)   # K % 64 != 0
