"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Q8_1 planes and sub-block integer sums must match bit for bit; fp32 outputs
must satisfy |y - y_oracle| <= 1e-4 * sum_k |w*xq| per element.  Small
shapes are compared on every output; the full-size shapes of the workloads
(27B-class layer, small-model decode with its LM head, chunked prefill,
512-token prefill) run in the same launch configuration the benchmark uses and
are compared on sampled rows (every 61st row and the last, all tokens).
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


def q8_from_oracle(qs, d, s) -> zq.Q8_1:
    return zq.Q8_1(to_dev(qs), to_dev(d.view(np.float16)), to_dev(s.view(np.float16)))


def q8_to_np(a: zq.Q8_1):
    torch.cuda.synchronize()
    return (a.qs.cpu().numpy(), a.d.cpu().numpy().view(np.uint16), a.s.cpu().numpy().view(np.uint16))


# ------------------------------------------------------------ RMSNorm + Q8_1
RMS_SHAPES = [(1, 32), (1, 96), (1, 1024), (1, 5120), (1, 6144), (1, 17408), (3, 8224),
              (4, 17408), (16, 5120), (2, 76800), (512, 5120), (512, 17408),
              # rows that are not whole groups of eight blocks, many tokens:
              # the staged kernel (545 blocks) and the thread-per-block one
              # (577 blocks: too wide for the staged kernel, not K % 256 for
              # the row-staged one)
              (6, 17440), (6, 18464), (40, 1056)]


@pytest.mark.parametrize("B,K", RMS_SHAPES)
def test_rmsnorm_q8_1_bit_exact(B, K):
    x = inputs.activations(100 + K, B, K)
    g = inputs.gamma(100 + K, K)
    ref = oracle_q8(x, g)
    got = q8_to_np(zq.rmsnorm_q8_1(to_dev(x), to_dev(g), inputs.EPS))
    for name, a, b in zip(("qs", "d", "s"), got, ref):
        assert np.array_equal(a, b), f"{name} differs at {np.argwhere(a != b)[:5].tolist()}"


def test_rmsnorm_q8_1_edge_cases():
    K = 512
    x = inputs.activations(5, 4, K)
    g = inputs.gamma(5, K)
    x[0] = 0.0                       # all-zero token: mean 0, r = 1/sqrt(eps), all blocks amax 0
    g2 = g.copy()
    g2[32:64] = 0.0                  # a block whose normalised values are all zero
    x[2, :] = 1.0                    # eps = 0 crafted ties through gamma
    g2[256:264] = [127.0, 2.5, -2.5, 1.5, -1.5, 0.5, -0.5, 63.5]
    x[3, 7] = 3e4                    # one huge outlier
    for eps in (inputs.EPS, 0.0, 0.5):
        xx = x.copy()
        if eps == 0.0:
            xx[0] = 1.0              # avoid 1/sqrt(0)
        ref = oracle_q8(xx, g2, eps)
        got = q8_to_np(zq.rmsnorm_q8_1(to_dev(xx), to_dev(g2), eps))
        for name, a, b in zip(("qs", "d", "s"), got, ref):
            assert np.array_equal(a, b), (eps, name)


# ------------------------------------------------------------ projections
def run_gemv(W, N, K, a):
    y = zq.q4k_gemv(to_dev(W), N, K, a)
    torch.cuda.synchronize()
    return y.cpu().numpy()[None, :]


GEMV_SHAPES = [  # (K, N): config-0 tile, ragged N, ragged super-block counts
    (1024, 1024), (256, 1), (256, 77), (768, 1000), (1280, 333), (3072, 1024), (2048, 1024),
    (32768, 1500)]   # the staging limit with full-size stages: shared memory at its maximum


@pytest.mark.parametrize("K,N", GEMV_SHAPES)
def test_gemv_all_rows(K, N):
    x, g, W = make_layer_inputs(K + N, 1, K, N)
    qs, d, s = oracle_q8(x, g)
    y_ref, S = oracle.q4k_matmul(W, N, K, qs, d, s)
    y = run_gemv(W, N, K, q8_from_oracle(qs, d, s))
    assert_within(y, y_ref, S, f"gemv K={K} N={N}")


@pytest.mark.parametrize("name,K,N,paired", inputs.LAYER_27B + inputs.SMALL_DECODE[:-1])
def test_decode_shapes_full(name, K, N, paired):
    """Every row of each decode projection (27B-class layer, small model)."""
    x, g, W = make_layer_inputs(7, 1, K, N)
    qs, d, s = oracle_q8(x, g)
    a = q8_from_oracle(qs, d, s)
    if paired:
        W2 = inputs.q4k_weights(7, N, K, tag_offset=100)
        yg, yu = zq.q4k_gemv_pair(to_dev(W), to_dev(W2), N, K, a)
        torch.cuda.synchronize()
        rg, Sg = oracle.q4k_matmul(W, N, K, qs, d, s)
        ru, Su = oracle.q4k_matmul(W2, N, K, qs, d, s)
        assert_within(yg.cpu().numpy()[None], rg, Sg, f"{name} gate")
        assert_within(yu.cpu().numpy()[None], ru, Su, f"{name} up")
    else:
        y_ref, S = oracle.q4k_matmul(W, N, K, qs, d, s)
        assert_within(run_gemv(W, N, K, a), y_ref, S, name)


def test_lm_head_sampled():
    K, N = 1024, 151936
    x, g, W = make_layer_inputs(8, 1, K, N)
    qs, d, s = oracle_q8(x, g)
    y = run_gemv(W, N, K, q8_from_oracle(qs, d, s))
    rows = sample_rows(N, 17)
    y_ref, S = oracle.q4k_matmul(W, N, K, qs, d, s, rows=rows)
    assert_within(y[:, rows], y_ref, S, "lm_head")


def test_gemv_pair_small_ragged():
    K, N = 768, 203
    x, g, W = make_layer_inputs(9, 1, K, N)
    W2 = inputs.q4k_weights(9, N, K, tag_offset=100)
    qs, d, s = oracle_q8(x, g)
    yg, yu = zq.q4k_gemv_pair(to_dev(W), to_dev(W2), N, K, q8_from_oracle(qs, d, s))
    torch.cuda.synchronize()
    for y, WW in ((yg, W), (yu, W2)):
        y_ref, S = oracle.q4k_matmul(WW, N, K, qs, d, s)
        assert_within(y.cpu().numpy()[None], y_ref, S, "pair")


def test_gemv_zero_activations_exact_zero():
    K, N = 512, 64
    _, _, W = make_layer_inputs(10, 1, K, N)
    x = np.zeros((1, K), np.float32)
    qs, d, s = oracle_q8(x, np.ones(K, np.float32))
    y = run_gemv(W, N, K, q8_from_oracle(qs, d, s))
    assert np.all(y == 0.0)


# ------------------------------------------------------------ integer sums
@pytest.mark.parametrize("B,K,N", [(1, 256, 5), (1, 1280, 37), (3, 512, 19)])
def test_isums_dp4a_bit_exact(B, K, N):
    x, g, W = make_layer_inputs(11 + B, B, K, N)
    qs, d, s = oracle_q8(x, g)
    I = zq.debug_q4k_isums(to_dev(W), N, K, q8_from_oracle(qs, d, s), path=0)
    torch.cuda.synchronize()
    assert np.array_equal(I.cpu().numpy(), oracle.q4k_isums(W, N, K, qs))


@pytest.mark.parametrize("B,K,N", [(17, 256, 128), (130, 512, 200), (256, 1024, 256), (128, 768, 77)])
def test_isums_tensor_core_bit_exact(B, K, N):
    """The tensor-core path's per-sub-block sums, read back from TMEM, equal
    the exact integer sums: fp16 operands and fp32 accumulation lose nothing."""
    x, g, W = make_layer_inputs(50 + B, B, K, N)
    qs, d, s = oracle_q8(x, g)
    I = zq.debug_q4k_isums(to_dev(W), N, K, q8_from_oracle(qs, d, s), path=1)
    torch.cuda.synchronize()
    assert zq.device_status() == 0
    assert np.array_equal(I.cpu().numpy(), oracle.q4k_isums(W, N, K, qs))


@pytest.mark.parametrize("B,K,N", [(2, 256, 64), (4, 512, 130), (16, 1280, 200)])
def test_isums_chunk_path_bit_exact(B, K, N):
    x, g, W = make_layer_inputs(60 + B, B, K, N)
    qs, d, s = oracle_q8(x, g)
    I = zq.debug_q4k_isums(to_dev(W), N, K, q8_from_oracle(qs, d, s), path=2)
    torch.cuda.synchronize()
    assert np.array_equal(I.cpu().numpy(), oracle.q4k_isums(W, N, K, qs))


def test_isums_extreme_codes_exact():
    """Largest magnitudes: q4 = 15, sc = 63, q8 = +-127 -> |sc*I| = 63*60960."""
    B, K, N = 128, 512, 128
    f = inputs.q4k_fields(70, N, K)
    f.q[...] = 15
    f.sc[...] = 63
    W = inputs.pack_q4k(f)
    qs = np.where(np.arange(B * K).reshape(B, K) % 3 == 0, -127, 127).astype(np.int8)
    qs[::2] = 127
    d = np.full((B, K // 32), 0x2008, np.uint16)
    s = np.full((B, K // 32), 0x3C00, np.uint16)
    I = zq.debug_q4k_isums(to_dev(W), N, K, q8_from_oracle(qs, d, s), path=1)
    torch.cuda.synchronize()
    assert np.array_equal(I.cpu().numpy(), oracle.q4k_isums(W, N, K, qs))
    y = run_gemm(W, N, K, q8_from_oracle(qs, d, s), B)
    y_ref, S = oracle.q4k_matmul(W, N, K, qs, d, s)
    assert_within(y, y_ref, S, "extreme codes")


# ------------------------------------------------------------ batched GEMM
def run_gemm(W, N, K, a, B):
    y = zq.q4k_gemm(to_dev(W), N, K, a, B)
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("B,K,N", [(2, 512, 50), (3, 2048, 257), (4, 1024, 129), (4, 17408, 40), (5, 768, 64), (8, 256, 300),
                                   (16, 1280, 130), (17, 512, 96), (130, 768, 200), (256, 1024, 256)])
def test_gemm_small_all_outputs(B, K, N):
    x, g, W = make_layer_inputs(20 + B, B, K, N)
    qs, d, s = oracle_q8(x, g)
    y = run_gemm(W, N, K, q8_from_oracle(qs, d, s), B)
    y_ref, S = oracle.q4k_matmul(W, N, K, qs, d, s)
    assert_within(y, y_ref, S, f"gemm B={B} K={K} N={N}")


@pytest.mark.parametrize("B,K,N", [(17, 1280, 77), (5, 1280, 65), (9, 2560, 131), (130, 1280, 203)])
def test_gemm_split_k_ragged_all_outputs(B, K, N):
    """Split-K launches whose output size B*N is not a multiple of four: every
    split's partial sums start on a 16-byte boundary and the reduction covers
    the last ragged group; every output against the oracle."""
    x, g, W = make_layer_inputs(25 + B, B, K, N)
    qs, d, s = oracle_q8(x, g)
    y = run_gemm(W, N, K, q8_from_oracle(qs, d, s), B)
    y_ref, S = oracle.q4k_matmul(W, N, K, qs, d, s)
    assert_within(y, y_ref, S, f"split-K gemm B={B} K={K} N={N}")


@pytest.mark.parametrize("B", inputs.CHUNK_BATCHES)
@pytest.mark.parametrize("name,K,N,paired", inputs.CHUNK_SHAPES)
def test_chunk_prefill_sampled(B, name, K, N, paired):
    x, g, W = make_layer_inputs(30 + B, B, K, N)
    qs, d, s = oracle_q8(x, g)
    y = run_gemm(W, N, K, q8_from_oracle(qs, d, s), B)
    rows = sample_rows(N)
    y_ref, S = oracle.q4k_matmul(W, N, K, qs, d, s, rows=rows)
    assert_within(y[:, rows], y_ref, S, f"chunk {name} B={B}")


@pytest.mark.parametrize("name,K,N,paired", inputs.LAYER_27B)
def test_prefill_512_sampled(name, K, N, paired):
    B = inputs.PREFILL_B
    x, g, W = make_layer_inputs(40, B, K, N)
    qs, d, s = oracle_q8(x, g)
    y = run_gemm(W, N, K, q8_from_oracle(qs, d, s), B)
    rows = sample_rows(N, 61 if N >= 4096 else 13)
    y_ref, S = oracle.q4k_matmul(W, N, K, qs, d, s, rows=rows)
    assert_within(y[:, rows], y_ref, S, f"prefill {name}")
