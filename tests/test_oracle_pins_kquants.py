"""Pins of the oracle's Q5_K and Q6_K functions against facts outside it.

The layouts are the readings stated in the oracle's header (the pages name
the formats -- MIInfer README, "Status": Q5_K x Q8_1 recurrent output
projection, MMVQ-style Q6_K x Q8_1 LM head -- but print no byte layout).
Pins: hand-worked blocks (tests/golden/hand_examples.json, derivations
there), round trips against the generator's vectorised packing, closed forms
of degenerate weights (pure fifth bit, Q6_K offset-only, single spike) and
brute force fp64 dequantise-then-matmul from the generator's fields.
"""
import json
import os

import numpy as np

import oracle
from gemm_zq_rmsnorm_gb300 import inputs

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "hand_examples.json")))


def f16(bits):
    return np.asarray(bits, np.uint16).view(np.float16).astype(np.float64)


def _q8(seed, B, K):
    x = inputs.activations(seed, B, K)
    return oracle.rmsnorm_q8_1(x, inputs.gamma(seed, K), inputs.EPS)


# ---------------------------------------------------------------- Q5_K
def test_q5k_unpack_hand_block():
    g4, g = GOLD["q4k_block"], GOLD["q5k_block"]
    blk = np.zeros(176, np.uint8)
    blk[0:4] = [int(b, 16) for b in g4["header"]]
    blk[4:16] = [int(b, 16) for b in g4["scale_bytes"]]
    for i in range(32):
        blk[16 + i] = 1 << (i % 8)
    for p in range(4):
        for i in range(32):
            blk[48 + 32 * p + i] = (i % 16) | (((p + i) % 16) << 4)
    d, dmin, sc, m, q = oracle.q5k_unpack(blk)
    assert d == np.float32(g4["d"]) and dmin == np.float32(g4["dmin"])
    assert sc.tolist() == g4["sc"] and m.tolist() == g4["m"]
    q = q.reshape(8, 32)
    for j, i, v in g["q"]:
        assert q[j, i] == v, (j, i)
    for p in range(4):
        for i in range(32):
            assert q[2 * p, i] == i % 16 + 16 * (i % 8 == 2 * p)
            assert q[2 * p + 1, i] == (p + i) % 16 + 16 * (i % 8 == 2 * p + 1)
    w = oracle.kq_dequant("q5k", blk, 1, 256).reshape(8, 32)
    for j, i, v in g["w"]:
        assert w[j, i] == v, (j, i)


def test_q5k_pack_unpack_roundtrip():
    N, K = 6, 768
    f = inputs.q5k_fields(12, N, K)
    W = inputs.pack_q5k(f).reshape(N, K // 256, 176)
    for n in range(N):
        for b in range(K // 256):
            d, dmin, sc, m, q = oracle.q5k_unpack(W[n, b])
            assert d == f16(f.d[n, b]) and dmin == f16(f.dmin[n, b])
            assert np.array_equal(sc, f.sc[n, b]) and np.array_equal(m, f.m[n, b])
            assert np.array_equal(q.reshape(8, 32), f.q[n, b])


def test_q5k_extreme_fields_roundtrip():
    N, K = 64, 256
    f = inputs.q5k_fields(6, N, K)
    f.sc[:, 0, :] = (np.arange(64)[:, None] + np.arange(8)[None, :] * 9) % 64
    f.m[:, 0, :] = 63 - f.sc[:, 0, :]
    f.q[::2] = 31
    f.q[1::2] = 0
    f.q[3::4, :, 5, :] = 16      # the fifth bit alone
    W = inputs.pack_q5k(f)
    for n in range(N):
        d, dmin, sc, m, q = oracle.q5k_unpack(W[n])
        assert np.array_equal(sc, f.sc[n, 0]) and np.array_equal(m, f.m[n, 0])
        assert np.array_equal(q.reshape(8, 32), f.q[n, 0])


def test_q5k_dequant_matches_fields():
    N, K = 4, 512
    f = inputs.q5k_fields(3, N, K)
    w = oracle.kq_dequant("q5k", inputs.pack_q5k(f), N, K)
    ref = (f16(f.d)[:, :, None, None] * f.sc[:, :, :, None] * f.q
           - f16(f.dmin)[:, :, None, None] * f.m[:, :, :, None]).reshape(N, K)
    assert np.array_equal(w, ref)


def test_q5k_fifth_bit_only_closed_form():
    """q = 16 everywhere: I_j = 16 * sum(q8) over the sub-block, so
    y = sum_b sum_j (16 d sc_j d8 sum(q8) - dmin m_j s8), same order as the
    definition (fp64, then one rounding to fp32)."""
    B, N, K = 2, 3, 512
    f = inputs.q5k_fields(7, N, K)
    f.q[...] = 16
    qs, d, s = _q8(7, B, K)
    y, _ = oracle.kq_matmul("q5k", inputs.pack_q5k(f), N, K, qs, d, s)
    qsum = qs.reshape(B, K // 32, 32).astype(np.int64).sum(-1)
    for t in range(B):
        for n in range(N):
            ref = 0.0
            for b in range(K // 256):
                for j in range(8):
                    c = 8 * b + j
                    ref += (f16(f.d[n, b]) * f.sc[n, b, j] * f16(d[t, c]) * float(16 * qsum[t, c])
                            - f16(f.dmin[n, b]) * f.m[n, b, j] * f16(s[t, c]))
            assert y[t, n] == np.float32(ref)


def test_q5k_equals_q4k_when_fifth_bit_clear():
    """With every fifth bit clear a Q5_K matrix is the Q4_K matrix of the same
    fields (an independent function of the oracle, pinned on its own)."""
    B, N, K = 2, 5, 512
    f = inputs.q5k_fields(8, N, K)
    f.q &= 15
    qs, d, s = _q8(8, B, K)
    y5, S5 = oracle.kq_matmul("q5k", inputs.pack_q5k(f), N, K, qs, d, s)
    f4 = inputs.Q4KFields(d=f.d, dmin=f.dmin, sc=f.sc, m=f.m, q=f.q)
    y4, S4 = oracle.q4k_matmul(inputs.pack_q4k(f4), N, K, qs, d, s)
    assert np.array_equal(y5, y4) and np.array_equal(S5, S4)


def test_q5k_matmul_brute_force_tiny():
    for (B, N, K, seed) in [(1, 1, 256, 30), (3, 7, 512, 31), (2, 4, 768, 32)]:
        f = inputs.q5k_fields(seed, N, K)
        qs, d, s = _q8(seed, B, K)
        y, S = oracle.kq_matmul("q5k", inputs.pack_q5k(f), N, K, qs, d, s)
        w = (f16(f.d)[:, :, None, None] * f.sc[:, :, :, None] * f.q
             - f16(f.dmin)[:, :, None, None] * f.m[:, :, :, None]).reshape(N, K)
        xq = (f16(d)[:, :, None] * qs.reshape(B, K // 32, 32)).reshape(B, K)
        y_bf = xq @ w.T
        S_bf = np.abs(xq[:, None, :] * w[None, :, :]).sum(-1)
        qsum = qs.reshape(B, K // 32, 32).astype(np.int64).sum(-1)
        sgap = np.abs(f16(s) - f16(d) * qsum)
        mins = (f16(f.dmin)[:, :, None] * f.m).reshape(N, K // 32)
        bound = sgap @ mins.T + 1e-12 * S_bf + np.abs(y_bf) * 2.0 ** -23
        assert np.all(np.abs(y - y_bf) <= bound)
        assert np.allclose(S, S_bf, rtol=1e-12, atol=0)


# ---------------------------------------------------------------- Q6_K
def _q6k_hand_block():
    g = GOLD["q6k_block"]
    blk = np.zeros(210, np.uint8)
    blk[0:64] = 0x21
    blk[64:128] = 0x53
    blk[128:160] = 0xE4
    blk[160:192] = 0x1B
    blk[192:208] = np.array(g["scales"], np.int8).view(np.uint8)
    blk[208:210] = [int(b, 16) for b in g["d_bytes"]]
    return blk


def test_q6k_unpack_hand_block():
    g = GOLD["q6k_block"]
    d, sc, q = oracle.q6k_unpack(_q6k_hand_block())
    assert d == np.float32(g["d"]) and sc.tolist() == g["scales"]
    for h in range(2):
        for c in range(4):
            assert np.all(q[128 * h + 32 * c: 128 * h + 32 * c + 32] == g["q_by_half_quarter"][h][c]), (h, c)
    w = oracle.kq_dequant("q6k", _q6k_hand_block(), 1, 256)[0]
    for k, v in g["w"]:
        assert w[k] == v, k


def test_q6k_pack_unpack_roundtrip():
    N, K = 6, 768
    f = inputs.q6k_fields(13, N, K)
    W = inputs.pack_q6k(f).reshape(N, K // 256, 210)
    for n in range(N):
        for b in range(K // 256):
            d, sc, q = oracle.q6k_unpack(W[n, b])
            assert d == f16(f.d[n, b])
            assert np.array_equal(sc, f.sc[n, b])
            assert np.array_equal(q.reshape(16, 16), f.q[n, b])


def test_q6k_extreme_fields_roundtrip():
    N, K = 64, 256
    f = inputs.q6k_fields(9, N, K)
    f.sc[:, 0, :] = ((np.arange(64)[:, None] * 4 + np.arange(16)[None, :] * 17) % 256 - 128).astype(np.int8)
    f.sc[0, 0, :] = -128
    f.sc[1, 0, :] = 127
    f.q[::2] = 63
    f.q[1::2] = 0
    f.q[3::4, :, 7, :] = 32
    W = inputs.pack_q6k(f)
    for n in range(N):
        d, sc, q = oracle.q6k_unpack(W[n])
        assert np.array_equal(sc, f.sc[n, 0])
        assert np.array_equal(q.reshape(16, 16), f.q[n, 0])


def test_q6k_dequant_matches_fields():
    N, K = 4, 512
    f = inputs.q6k_fields(3, N, K)
    w = oracle.kq_dequant("q6k", inputs.pack_q6k(f), N, K)
    ref = (f16(f.d)[:, :, None, None] * f.sc.astype(np.float64)[:, :, :, None]
           * (f.q.astype(np.float64) - 32)).reshape(N, K)
    assert np.array_equal(w, ref)


def test_q6k_offset_only_is_zero():
    """q = 32 everywhere encodes zero weights: y is exactly 0 and S is 0."""
    B, N, K = 2, 3, 512
    f = inputs.q6k_fields(10, N, K)
    f.q[...] = 32
    qs, d, s = _q8(10, B, K)
    y, S = oracle.kq_matmul("q6k", inputs.pack_q6k(f), N, K, qs, d, s)
    assert np.all(y == 0) and np.all(S == 0)


def test_q6k_single_spike():
    """One non-zero weight: q = 63 at k0 (all else 32), sc = -128 there, and one
    activation spike at k0: I = 31 * 127 and y = d * sc * d8 * I exactly."""
    k0 = 77
    f = inputs.q6k_fields(11, 1, 256)
    f.q[...] = 32
    f.q[0, 0, k0 // 16, k0 % 16] = 63
    f.sc[0, 0, k0 // 16] = -128
    f.d[0, 0] = 0x1400                      # 2^-10
    x = np.zeros((1, 256), np.float32)
    x[0, k0] = 16.0
    qs, d, s = oracle.rmsnorm_q8_1(x, np.ones(256, np.float32), 0.0)
    assert qs[0, k0] == 127 and np.count_nonzero(qs) == 1
    y, S = oracle.kq_matmul("q6k", inputs.pack_q6k(f), 1, 256, qs, d, s)
    ref = 2.0 ** -10 * -128 * f16(d[0, k0 // 32]) * (31 * 127)
    assert float(y[0, 0]) == np.float32(ref) and S[0, 0] == abs(ref)


def test_q6k_matmul_brute_force_tiny():
    for (B, N, K, seed) in [(1, 1, 256, 40), (3, 7, 512, 41), (2, 5, 1024, 42)]:
        f = inputs.q6k_fields(seed, N, K)
        qs, d, s = _q8(seed, B, K)
        y, S = oracle.kq_matmul("q6k", inputs.pack_q6k(f), N, K, qs, d, s)
        w = (f16(f.d)[:, :, None, None] * f.sc.astype(np.float64)[:, :, :, None]
             * (f.q.astype(np.float64) - 32)).reshape(N, K)
        xq = (f16(d)[:, :, None] * qs.reshape(B, K // 32, 32)).reshape(B, K)
        y_bf = xq @ w.T
        S_bf = np.abs(xq[:, None, :] * w[None, :, :]).sum(-1)
        # no min term: only fp64 summation order and the final fp32 rounding differ
        assert np.all(np.abs(y - y_bf) <= 1e-12 * S_bf + np.abs(y_bf) * 2.0 ** -23)
        assert np.allclose(S, S_bf, rtol=1e-12, atol=0)


def test_kq_row_subset_matches_full():
    B, N, K = 2, 9, 512
    qs, d, s = _q8(21, B, K)
    for fmt, W in (("q5k", inputs.q5k_weights(21, N, K)), ("q6k", inputs.q6k_weights(21, N, K))):
        y, S = oracle.kq_matmul(fmt, W, N, K, qs, d, s)
        rows = [8, 0, 4]
        ys, Ss = oracle.kq_matmul(fmt, W, N, K, qs, d, s, rows=rows)
        assert np.array_equal(ys, y[:, rows]) and np.array_equal(Ss, S[:, rows])
