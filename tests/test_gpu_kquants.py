"""GPU parity of the Q5_K and Q6_K projections against the oracle.

Small shapes are compared on every output (several tiles per CTA, ragged
row counts, a Q6_K matrix whose byte length is not a multiple of 16 so the
last tile's tail goes through the plain-load path, rows split into pieces at
K = 32768); the full-size workload shapes (the LM head 1024 -> 151936 in Q6_K,
the recurrent output projection 6144 -> 5120 in Q5_K at B = 1 and 4) run in
the benchmark's launch configuration and are compared on sampled rows.  The
fused RMSNorm + Q6_K mat-vec must reproduce the Q8_1 bytes of the oracle and
the two-step result bit for bit.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import gemm_zq_rmsnorm_gb300 as zq
from gemm_zq_rmsnorm_gb300 import inputs

from _cases import assert_within, oracle_q8, sample_rows

pytestmark = pytest.mark.gpu

DEV = "cuda"
WEIGHTS = {"q5k": inputs.q5k_weights, "q6k": inputs.q6k_weights}


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def q8_dev(qs, d, s) -> zq.Q8_1:
    return zq.Q8_1(to_dev(qs), to_dev(d.view(np.float16)), to_dev(s.view(np.float16)))


def run(fmt, W, N, K, q8):
    y = zq.kq_gemm(fmt, to_dev(W), N, K, q8_dev(*q8))
    torch.cuda.synchronize()
    return y.cpu().numpy()


SMALL = [  # (N, K, B)
    (1, 256, 1), (7, 256, 1), (7, 256, 3), (300, 768, 1), (300, 768, 4), (300, 768, 5),
    (513, 1024, 2), (129, 2816, 16), (1000, 5120, 1), (64, 5120, 8), (5, 32768, 1), (5, 32768, 4),
    (3, 32768, 6), (70, 29696, 4)]   # 29696: the largest K whose four-token Q6_K staging fits


@pytest.mark.parametrize("fmt", ["q5k", "q6k"])
@pytest.mark.parametrize("N,K,B", SMALL)
def test_kq_small_all_outputs(fmt, N, K, B):
    seed = 7 * N + K + B
    W = WEIGHTS[fmt](seed, N, K)
    assert W.nbytes == zq.kq_bytes(fmt, N, K)
    q8 = oracle_q8(inputs.activations(seed, B, K), inputs.gamma(seed, K))
    y_ref, S = oracle.kq_matmul(fmt, W, N, K, *q8)
    y = run(fmt, W, N, K, q8)
    assert y.shape == (B, N)
    assert_within(y, y_ref, S, f"{fmt} {N}x{K} B={B}")


@pytest.mark.parametrize("fmt", ["q5k", "q6k"])
def test_kq_tokens_independent(fmt):
    """A token's result does not depend on which launch group it falls in."""
    N, K, B = 200, 1024, 9
    W = WEIGHTS[fmt](3, N, K)
    qs, d, s = oracle_q8(inputs.activations(3, B, K), inputs.gamma(3, K))
    y_all = run(fmt, W, N, K, (qs, d, s))
    for t in (0, 4, 8):
        y_one = run(fmt, W, N, K, (qs[t:t + 1], d[t:t + 1], s[t:t + 1]))
        assert np.array_equal(y_one[0], y_all[t])


@pytest.mark.parametrize("fmt", ["q5k", "q6k"])
def test_kq_degenerate_weights(fmt):
    """All-zero activations give y = 0 exactly; Q6_K with every q = 32 (zero
    weights) gives 0 for any input."""
    N, K = 96, 512
    W = WEIGHTS[fmt](4, N, K)
    B = 2
    qs = np.zeros((B, K), np.int8)
    d = np.zeros((B, K // 32), np.uint16)
    s = np.zeros((B, K // 32), np.uint16)
    assert np.all(run(fmt, W, N, K, (qs, d, s)) == 0.0)
    if fmt == "q6k":
        f = inputs.q6k_fields(4, N, K)
        f.q[...] = 32
        q8 = oracle_q8(inputs.activations(4, B, K), inputs.gamma(4, K))
        assert np.all(run(fmt, inputs.pack_q6k(f), N, K, q8) == 0.0)


def test_q6k_lm_head_sampled():
    """Q6_K LM head of the small model, 1024 -> 151936, B = 1."""
    N, K = 151936, 1024
    W = inputs.q6k_weights(0, N, K, tag_offset=600)
    q8 = oracle_q8(inputs.activations(0, 1, K), inputs.gamma(0, K))
    y = run("q6k", W, N, K, q8)
    rows = sample_rows(N)
    y_ref, S = oracle.kq_matmul("q6k", W, N, K, *q8, rows=rows)
    assert_within(y[:, rows], y_ref, S, "q6k lm_head")


@pytest.mark.parametrize("B", [1, 4])
def test_q5k_recurrent_out_sampled(B):
    """Q5_K recurrent output projection of the 27B-class layer, 6144 -> 5120."""
    N, K = 5120, 6144
    W = inputs.q5k_weights(0, N, K, tag_offset=500)
    q8 = oracle_q8(inputs.activations(B, B, K), inputs.gamma(0, K))
    y = run("q5k", W, N, K, q8)
    rows = sample_rows(N)
    y_ref, S = oracle.kq_matmul("q5k", W, N, K, *q8, rows=rows)
    assert_within(y[:, rows], y_ref, S, f"q5k 6144->5120 B={B}")


@pytest.mark.parametrize("N,K", [(7, 256), (4001, 1024), (2048, 5120)])
def test_rmsnorm_q6k_gemv_fused(N, K):
    x = inputs.activations(11 + N, 1, K)
    g = inputs.gamma(11, K)
    W = inputs.q6k_weights(11, N, K)
    ref_q8 = oracle_q8(x, g)
    Wd = to_dev(W)
    q8_out = zq.empty_q8_1(1, K)
    y = zq.rmsnorm_q6k_gemv(to_dev(x[0]), to_dev(g), inputs.EPS, Wd, N, q8_out=q8_out)
    y2 = zq.kq_gemm("q6k", Wd, N, K, zq.rmsnorm_q8_1(to_dev(x), to_dev(g), inputs.EPS))
    torch.cuda.synchronize()
    got_q8 = (q8_out.qs.cpu().numpy(), q8_out.d.cpu().numpy().view(np.uint16),
              q8_out.s.cpu().numpy().view(np.uint16))
    for name, a, b in zip(("qs", "d", "s"), got_q8, ref_q8):
        assert np.array_equal(a, b), name
    assert np.array_equal(y.cpu().numpy(), y2.cpu().numpy()[0])
    y_ref, S = oracle.kq_matmul("q6k", W, N, K, *ref_q8)
    assert_within(y.cpu().numpy()[None, :], y_ref, S, f"fused rmsnorm+q6k {N}x{K}")


def test_kq_rejects():
    W = torch.zeros(zq.kq_bytes("q6k", 8, 512) + 16, dtype=torch.uint8, device=DEV)
    a = zq.empty_q8_1(17, 512)
    y = torch.empty((17, 8), dtype=torch.float32, device=DEV)
    with pytest.raises(zq.ZQError) as e:
        zq.kq_gemm("q6k", W, 8, 512, a, B=17, y=y)
    assert e.value.status == -2
    with pytest.raises(zq.ZQError) as e:
        zq.kq_gemm("q5k", W[1:], 8, 512, a.rows(0, 1), y=y[0])
    assert e.value.status == -3
