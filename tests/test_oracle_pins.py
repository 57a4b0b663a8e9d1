"""Pins of the CPU oracle against facts that do not come from the oracle.

Each test ties one oracle function to something fixed outside it: a
hand-worked example (values derived by hand in the comments and stored in
tests/golden/hand_examples.json), a closed form, a library routine for a
special case (numpy's binary16 conversion), or brute force on tiny shapes
computed from the generator's unpacked fields (never from the oracle's own
unpacking).  A dropped term, a wrong sign, a swapped nibble or a transposed
index in the oracle fails at least one of them.
"""
import json
import os

import numpy as np
import pytest

import oracle
from gemm_zq_rmsnorm_gb300 import inputs

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "hand_examples.json")))


def f16(bits):
    return np.asarray(bits, np.uint16).view(np.float16).astype(np.float64)


# ---------------------------------------------------------------- binary16
def test_f16_hand_values():
    for v, h in GOLD["f16"]:
        assert int(oracle.f32_to_f16_bits([np.float32(v)])[0]) == int(h, 16), v


def test_f16_matches_numpy_boundaries_and_random():
    # every power of two across the range, and points around the rounding
    # boundaries of each binade (midpoints, +-1 ulp of fp32)
    vals = []
    for e in range(-26, 17):
        base = np.float32(2.0 ** e)
        for frac in range(0, 1025, 7):
            v = np.float32((1.0 + frac / 1024.0) * 2.0 ** e)
            mid = np.float32((1.0 + (frac + 0.5) / 1024.0) * 2.0 ** e)
            vals += [v, mid, np.nextafter(mid, np.float32(0)), np.nextafter(mid, np.float32(np.inf)), base]
    vals += [65504.0, 65519.0, 65520.0, 65535.0, 1e9, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -25, 2.0 ** -26, 0.0]
    rng = np.random.default_rng(0)
    rb = rng.integers(0, 2 ** 32, 300_000, dtype=np.uint64).astype(np.uint32).view(np.float32)
    rb = rb[np.isfinite(rb)]
    v = np.concatenate([np.asarray(vals, np.float32), -np.asarray(vals, np.float32), rb])
    ours = oracle.f32_to_f16_bits(v)
    with np.errstate(over="ignore"):
        ref = v.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


def test_f16_decode_all_patterns():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.f16_bits_to_f32(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


# ---------------------------------------------------------------- Q4_K layout
def test_q4k_unpack_hand_block():
    g = GOLD["q4k_block"]
    blk = np.zeros(144, np.uint8)
    blk[0:4] = [int(b, 16) for b in g["header"]]
    blk[4:16] = [int(b, 16) for b in g["scale_bytes"]]
    # nibble byte 32p+i = (i % 16) | ((p + i) % 16) << 4
    for p in range(4):
        for i in range(32):
            blk[16 + 32 * p + i] = (i % 16) | (((p + i) % 16) << 4)
    d, dmin, sc, m, q = oracle.q4k_unpack(blk)
    assert d == np.float32(g["d"]) and dmin == np.float32(g["dmin"])
    assert sc.tolist() == g["sc"]
    assert m.tolist() == g["m"]
    q = q.reshape(8, 32)
    for p in range(4):
        assert q[2 * p].tolist() == [i % 16 for i in range(32)]
        assert q[2 * p + 1].tolist() == [(p + i) % 16 for i in range(32)]


def test_q4k_pack_unpack_roundtrip():
    N, K = 7, 768
    f = inputs.q4k_fields(11, N, K)
    W = inputs.pack_q4k(f).reshape(N, K // 256, 144)
    for n in range(N):
        for b in range(K // 256):
            d, dmin, sc, m, q = oracle.q4k_unpack(W[n, b])
            assert d == f16(f.d[n, b]) and dmin == f16(f.dmin[n, b])
            assert np.array_equal(sc, f.sc[n, b]) and np.array_equal(m, f.m[n, b])
            assert np.array_equal(q.reshape(8, 32), f.q[n, b])


def test_q4k_extreme_fields_roundtrip():
    # all 6-bit scale/min values in every slot, both nibble extremes
    N, K = 64, 256
    f = inputs.q4k_fields(5, N, K)
    f.sc[:, 0, :] = (np.arange(64)[:, None] + np.arange(8)[None, :] * 9) % 64
    f.m[:, 0, :] = 63 - f.sc[:, 0, :]
    f.q[::2] = 15
    f.q[1::2] = 0
    W = inputs.pack_q4k(f)
    for n in range(N):
        d, dmin, sc, m, q = oracle.q4k_unpack(W[n])
        assert np.array_equal(sc, f.sc[n, 0]) and np.array_equal(m, f.m[n, 0])
        assert np.array_equal(q.reshape(8, 32), f.q[n, 0])


def test_dequant_matches_fields():
    N, K = 5, 512
    f = inputs.q4k_fields(3, N, K)
    w = oracle.q4k_dequant(inputs.pack_q4k(f), N, K)
    ref = (f16(f.d)[:, :, None, None] * f.sc[:, :, :, None] * f.q
           - f16(f.dmin)[:, :, None, None] * f.m[:, :, :, None]).reshape(N, K)
    assert np.array_equal(w, ref)


# ---------------------------------------------------------------- RMSNorm
def test_rms_scale_exact_cases():
    rng = np.random.default_rng(1)
    for K in (256, 1024, 17408):
        x = rng.choice([-1.0, 1.0], K).astype(np.float32)
        assert oracle.rms_scale(x, 0.0) == np.float32(1.0)           # ss = K
        assert oracle.rms_scale(2 * x, 0.0) == np.float32(0.5)       # mean 4
    assert oracle.rms_scale(np.zeros(256, np.float32), 0.25) == np.float32(2.0)  # eps only
    assert oracle.rms_scale(np.full(512, 3.0, np.float32), 7.0) == np.float32(0.25)  # 9 + 7


def test_rms_scale_vs_fp64():
    rng = np.random.default_rng(2)
    for K in (256, 1024, 5120, 17408):
        x = inputs.activations(int(rng.integers(1 << 30)), 1, K)[0]
        r = oracle.rms_scale(x, 1e-6)
        r64 = 1.0 / np.sqrt(np.sum(x.astype(np.float64) ** 2) / K + 1e-6)
        assert abs(r - r64) <= 4e-7 * r64


def test_q8_1_crafted_block():
    g = GOLD["q8_1_block"]
    K = 256
    x = np.ones((1, K), np.float32)
    gamma = np.zeros(K, np.float32)
    gamma[: len(g["gamma0"])] = g["gamma0"]           # block 0: crafted values
    gamma[64:96] = 0.0                                # block 2: all zero
    gamma[96] = -6.0                                  # block 3: d = 6/127
    gamma[97] = 3.0
    gamma[98] = 1.0
    qs, d, s = oracle.rmsnorm_q8_1(x, gamma, 0.0)     # ss = K, r = 1, xh = gamma
    assert qs[0, :32].tolist() == g["q0"]
    assert d[0, 0] == int(g["d0"], 16) and s[0, 0] == int(g["s0"], 16)
    assert qs[0, 64:96].tolist() == [0] * 32 and d[0, 2] == 0 and s[0, 2] == 0
    # block 3: d = 6/127, q = round(xh*(127/6)): -127, 63.5 -> 64 (half away), 21.17 -> 21
    assert qs[0, 96:99].tolist() == [-127, 64, 21]
    assert d[0, 3] == np.float16(np.float32(6.0) / np.float32(127.0)).view(np.uint16)


def test_q8_1_properties_random():
    B, K = 3, 5120
    x = inputs.activations(7, B, K)
    gamma = inputs.gamma(7, K)
    qs, d, s = oracle.rmsnorm_q8_1(x, gamma, inputs.EPS)
    qb = qs.reshape(B, K // 32, 32).astype(np.int64)
    # each block reaches +-127 exactly at its largest |value|; codes in range
    assert np.all(np.abs(qb).max(-1) == 127)
    assert qb.min() >= -127 and qb.max() <= 127
    # s = fp16(d32 * sum q): |s16 - d16*sum| within two fp16 roundings
    ssum = qb.sum(-1).astype(np.float64)
    dd, ss_ = f16(d), f16(s)
    assert np.all(np.abs(ss_ - dd * ssum) <= (2.0 ** -10) * np.abs(dd * ssum) + 1e-7)
    # dequantised activations approximate the fp64 RMSNorm within half a step
    r = np.array([1.0 / np.sqrt(np.mean(x[t].astype(np.float64) ** 2) + inputs.EPS) for t in range(B)])
    xh = x.astype(np.float64) * r[:, None] * gamma.astype(np.float64)
    xq = (dd[:, :, None] * qb).reshape(B, K)
    step = np.repeat(dd, 32, axis=1)
    assert np.all(np.abs(xq - xh) <= 0.5 * step + 2e-3 * np.abs(xh) + 1e-6)


# ---------------------------------------------------------------- integer sums
def test_isums_brute_force():
    for (B, N, K, seed) in [(1, 3, 256, 0), (3, 8, 512, 1), (2, 5, 1024, 2)]:
        f = inputs.q4k_fields(seed, N, K)
        W = inputs.pack_q4k(f)
        x = inputs.activations(seed, B, K)
        qs, _, _ = oracle.rmsnorm_q8_1(x, inputs.gamma(seed, K), inputs.EPS)
        I = oracle.q4k_isums(W, N, K, qs)
        q4 = f.q.reshape(N, K).astype(np.int64)
        ref = np.einsum("nkc,tkc->tnk", q4.reshape(N, K // 32, 32),
                        qs.astype(np.int64).reshape(B, K // 32, 32))
        assert np.array_equal(I, ref)


# ---------------------------------------------------------------- the product
def _one_block_matrix(q_val, sc_val, m_val, d_bits, dmin_bits, K=256, N=1):
    f = inputs.q4k_fields(0, N, K)
    f.q[...] = q_val
    f.sc[...] = sc_val
    f.m[...] = m_val
    f.d[...] = d_bits
    f.dmin[...] = dmin_bits
    return f


def test_E1_all_ones():
    g = GOLD["E1"]
    f = _one_block_matrix(1, 1, 0, 0x3C00, 0x0000)
    x = np.full((1, 256), 1000.0, np.float32)
    qs, d, s = oracle.rmsnorm_q8_1(x, np.ones(256, np.float32), 1e-6)
    assert np.all(qs == 127) and np.all(d == int(g["d8"], 16))
    y, S = oracle.q4k_matmul(inputs.pack_q4k(f), 1, 256, qs, d, s)
    assert float(y[0, 0]) == g["y"]


def test_E2_zero_quants_closed_form():
    B, N, K = 2, 4, 512
    f = inputs.q4k_fields(4, N, K)
    f.q[...] = 0
    x = inputs.activations(4, B, K)
    qs, d, s = oracle.rmsnorm_q8_1(x, inputs.gamma(4, K), inputs.EPS)
    y, _ = oracle.q4k_matmul(inputs.pack_q4k(f), N, K, qs, d, s)
    nb = K // 256
    for t in range(B):
        for n in range(N):
            ref = 0.0
            for b in range(nb):
                for j in range(8):
                    ref -= f16(f.dmin[n, b]) * f.m[n, b, j] * f16(s[t, 8 * b + j])
            assert y[t, n] == np.float32(ref)


def test_E3_single_spike():
    g = GOLD["E3"]
    k0 = g["k0"]
    f = _one_block_matrix(0, 63, 0, 0x1400, 0x0000)   # d = 2^-10
    f.q[0, 0, k0 // 32, k0 % 32] = 15
    x = np.zeros((1, 256), np.float32)
    x[0, k0] = 16.0
    qs, d, s = oracle.rmsnorm_q8_1(x, np.ones(256, np.float32), 0.0)
    assert qs[0, k0] == 127 and np.count_nonzero(qs) == 1
    assert d[0, k0 // 32] == int(g["d8"], 16)
    others = [j for j in range(8) if j != k0 // 32]
    assert np.all(d[0, others] == 0) and np.all(s[0, others] == 0)
    I = oracle.q4k_isums(inputs.pack_q4k(f), 1, 256, qs)
    assert I[0, 0, k0 // 32] == 1905
    y, _ = oracle.q4k_matmul(inputs.pack_q4k(f), 1, 256, qs, d, s)
    assert float(y[0, 0]) == g["y_num"] / 2.0 ** g["y_pow2"]


def test_matmul_brute_force_tiny():
    for (B, N, K, seed) in [(1, 1, 256, 10), (3, 8, 512, 11), (2, 6, 256, 12), (1, 8, 512, 13)]:
        f = inputs.q4k_fields(seed, N, K)
        W = inputs.pack_q4k(f)
        x = inputs.activations(seed, B, K)
        qs, d, s = oracle.rmsnorm_q8_1(x, inputs.gamma(seed, K), inputs.EPS)
        y, S = oracle.q4k_matmul(W, N, K, qs, d, s)
        w = (f16(f.d)[:, :, None, None] * f.sc[:, :, :, None] * f.q
             - f16(f.dmin)[:, :, None, None] * f.m[:, :, :, None]).reshape(N, K)
        xq = (f16(d)[:, :, None] * qs.reshape(B, K // 32, 32)).reshape(B, K)
        y_bf = xq @ w.T
        S_bf = np.abs(xq[:, None, :] * w[None, :, :]).sum(-1)
        # the oracle uses s16 where brute force has d16*sum(q): bound that gap
        qsum = qs.reshape(B, K // 32, 32).astype(np.int64).sum(-1)
        sgap = np.abs(f16(s) - f16(d) * qsum)                            # [B, K/32]
        mins = (f16(f.dmin)[:, :, None] * f.m).reshape(N, K // 32)       # [N, K/32]
        bound = sgap @ mins.T + 1e-12 * S_bf + np.abs(y_bf) * 2.0 ** -23
        assert np.all(np.abs(y - y_bf) <= bound)
        assert np.allclose(S, S_bf, rtol=1e-12, atol=0)


def test_row_subset_matches_full():
    B, N, K = 2, 9, 512
    W = inputs.q4k_weights(21, N, K)
    x = inputs.activations(21, B, K)
    qs, d, s = oracle.rmsnorm_q8_1(x, inputs.gamma(21, K), inputs.EPS)
    y, S = oracle.q4k_matmul(W, N, K, qs, d, s)
    rows = [8, 0, 4]
    ys, Ss = oracle.q4k_matmul(W, N, K, qs, d, s, rows=rows)
    assert np.array_equal(ys, y[:, rows]) and np.array_equal(Ss, S[:, rows])


def test_dequant_f16_matches_numpy_float32_steps():
    """Binary16 weights: numpy's own IEEE float32 steps (a = d*sc, b = dmin*m,
    a*q - b) and its float16 rounding, from the generator's fields (not the
    oracle's unpacking)."""
    N, K = 3, 512
    f = inputs.q4k_fields(21, N, K)
    W = inputs.pack_q4k(f)
    got = oracle.q4k_dequant_f16(W, N, K)
    d = f.d.view(np.float16).astype(np.float32)      # [N][nb]
    dm = f.dmin.view(np.float16).astype(np.float32)
    nb = K // 256
    want = np.zeros((N, K), np.uint16)
    for n in range(N):
        for b in range(nb):
            for j in range(8):
                a = np.float32(d[n, b] * np.float32(f.sc[n, b, j]))
                bm = np.float32(dm[n, b] * np.float32(f.m[n, b, j]))
                q = f.q[n, b, j].astype(np.float32)
                w = (a * q - bm).astype(np.float32)
                want[n, 256 * b + 32 * j:256 * b + 32 * j + 32] = w.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, want)


def test_dequant_f16_within_half_ulp_of_fp64():
    """|w16 - w| <= half a binary16 ulp of w plus the fp32 rounding, against
    the fp64 dequantisation, on random and extreme fields."""
    N, K = 64, 1024
    W = inputs.q4k_weights(22, N, K)
    w64 = oracle.q4k_dequant(W, N, K)
    w16 = oracle.q4k_dequant_f16(W, N, K).view(np.float16).astype(np.float64)
    a = np.abs(w64)
    ulp16 = np.where(a < 2.0 ** -14, 2.0 ** -24, 2.0 ** (np.floor(np.log2(np.maximum(a, 2.0 ** -14))) - 10))
    assert np.all(np.abs(w16 - w64) <= 0.5 * ulp16 + a * 2.0 ** -24 + 1e-30)


# ------------------------------------------- dequantise-then-GEMM (binary16)
def test_q8_1_dequant_f16_hand_values():
    """x = q8 * d8 rounded to binary16, worked by hand:
    127 * 0.0625 = 7.9375 = 1.984375 * 2^2 -> 0x4400 | 1008 = 0x47F0 (exact);
    -127 * 0.0625 -> 0xC7F0;
    127 * (1 + 2^-10) = 127.1240234375, binary16 step 2^-4 in [64, 128):
      nearest is 127.125 = 1.986328125 * 2^6 -> 0x5400 | 1010 = 0x57F2;
    3 * (1 + 3 * 2^-10) = 3.0087890625 = 1540.5 steps of 2^-9: a tie, to the
      even 1540 -> 3.0078125 = 1.50390625 * 2 -> 0x4000 | 516 = 0x4204;
    1 * 2^-24 (the smallest subnormal d8) -> 0x0001; 0 * anything -> 0."""
    qs = np.zeros((1, 64), np.int8)
    d = np.zeros((1, 2), np.uint16)
    d[0, 0] = 0x2C00
    qs[0, 0], qs[0, 1] = 127, -127
    d[0, 1] = 0x3C01
    qs[0, 32] = 127
    got = oracle.q8_1_dequant_f16(qs, d)
    assert got[0, 0] == 0x47F0 and got[0, 1] == 0xC7F0 and got[0, 32] == 0x57F2
    assert np.all(got[0, 2:32] == 0) and np.all(got[0, 33:] == 0)
    qs2 = np.zeros((2, 32), np.int8)
    qs2[0, 5] = 3
    qs2[1, 7] = 1
    d2 = np.array([[0x3C03], [0x0001]], np.uint16)
    got2 = oracle.q8_1_dequant_f16(qs2, d2)
    assert got2[0, 5] == 0x4204 and got2[1, 7] == 0x0001
    assert np.count_nonzero(got2) == 2


def test_q8_1_dequant_f16_matches_numpy():
    """Random codes and scales: numpy's float32 product and float16 rounding,
    with the block index k // 32 taken per token."""
    rng = np.random.default_rng(5)
    B, K = 3, 256
    qs = rng.integers(-127, 128, size=(B, K)).astype(np.int8)
    d = (rng.random((B, K // 32)) * 0.05).astype(np.float16).view(np.uint16)
    want = (qs.astype(np.float32) * np.repeat(d.view(np.float16).astype(np.float32), 32, axis=1)).astype(
        np.float16).view(np.uint16)
    assert np.array_equal(oracle.q8_1_dequant_f16(qs, d), want)


def test_f16_gemm_brute_force_exact():
    """y = x w^T against exact rational sums on a tiny shape (distinct rows
    and tokens, so a transposed operand or a dropped term shows)."""
    from fractions import Fraction
    rng = np.random.default_rng(6)
    B, N, K = 2, 3, 64
    x = (rng.standard_normal((B, K)) * 4).astype(np.float16)
    w = (rng.standard_normal((N, K)) / 8).astype(np.float16)
    y = oracle.f16_gemm(x.view(np.uint16), w.view(np.uint16))
    for t in range(B):
        for n in range(N):
            exact = sum(Fraction(float(x[t, k])) * Fraction(float(w[n, k])) for k in range(K))
            assert abs(Fraction(y[t, n]) - exact) <= abs(exact) * Fraction(1, 2 ** 50) + Fraction(1, 2 ** 60)
    rows = [2, 0]
    assert np.array_equal(oracle.f16_gemm(x.view(np.uint16), w.view(np.uint16), rows=rows), y[:, rows])


def test_f16_gemm_selector_rows():
    """w with one 1 per row picks a column of x: y[t][n] = x[t][perm[n]]."""
    B, N, K = 4, 5, 64
    x = np.arange(B * K, dtype=np.float32).reshape(B, K).astype(np.float16) - 100
    perm = [7, 0, 63, 31, 2]
    w = np.zeros((N, K), np.float16)
    for n, k in enumerate(perm):
        w[n, k] = 1
    y = oracle.f16_gemm(x.view(np.uint16), w.view(np.uint16))
    assert np.array_equal(y, x.astype(np.float64)[:, perm])


# ---------------------------------------------------------------- SiLU * up
def test_exp32_within_two_ulp_of_fp64():
    """exp32 against numpy's fp64 exponential on a dense grid of the clamped
    range, and exactly 1 at 0."""
    a = np.concatenate([np.linspace(-86, 88, 200001), np.linspace(-1, 1, 20001)]).astype(np.float32)
    e = oracle.exp32(a).astype(np.float64)
    ref = np.exp(a.astype(np.float64))
    assert np.all(np.abs(e - ref) <= 2.0 ** -22 * ref)
    assert oracle.exp32([0.0])[0] == 1.0


def test_silu32_identities():
    """silu(0) = 0; silu(g) - silu(-g) = g (the two logistic factors sum to
    one); silu(g) -> g for large g and -> 0 for very negative g; within a
    few ulp of the fp64 formula."""
    g = np.linspace(-20, 20, 40001).astype(np.float32)
    s = oracle.silu32(g).astype(np.float64)
    sn = oracle.silu32(-g).astype(np.float64)
    gd = g.astype(np.float64)
    assert oracle.silu32([0.0])[0] == 0.0
    assert np.all(np.abs((s - sn) - gd) <= 1e-6 * np.maximum(np.abs(gd), 1e-30) + 1e-7)
    ref = gd / (1.0 + np.exp(-gd))
    assert np.all(np.abs(s - ref) <= 2.0 ** -21 * np.abs(ref) + 1e-30)
    big = oracle.silu32([30.0, 80.0, -80.0])
    assert big[0] == np.float32(30.0) and big[1] == np.float32(80.0) and abs(big[2]) < 1e-30


def test_silu_mul_q8_1_zero_up_and_single_spike():
    """up = 0 gives all-zero codes and scales; a single non-zero product in a
    block packs to code 127 with d = |h| / 127."""
    K = 64
    g = np.linspace(-3, 3, K, dtype=np.float32)[None]
    qs, d, s = oracle.silu_mul_q8_1(g, np.zeros((1, K), np.float32))
    assert not qs.any() and not d.any() and not s.any()
    u = np.zeros((1, K), np.float32)
    u[0, 40] = 2.0
    qs, d, s = oracle.silu_mul_q8_1(g, u)
    h = oracle.silu32([g[0, 40]])[0] * np.float32(2.0)
    assert qs[0, 40] == (127 if h > 0 else -127) and np.count_nonzero(qs) == 1
    d32 = np.float32(abs(h)) / np.float32(127.0)
    assert d[0, 1] == oracle.f32_to_f16_bits([d32])[0]
    # s = fp16(d32 * sum q): the one code is +-127
    assert s[0, 1] == oracle.f32_to_f16_bits([d32 * np.float32(127.0 if h > 0 else -127.0)])[0]
    # the other block holds no non-zero product: d = s = 0
    assert d[0, 0] == 0 and s[0, 0] == 0


def test_silu_mul_q8_1_hand_blocks():
    """Hand-derived blocks.  silu32(32) = 32 exactly (exp32(-32) < 2^-24, so
    1 + exp32(-32) rounds to 1), so with gate = 32 the product h = 32 * up is
    exact for dyadic up.  Block 0: h = 127, +-2.5, +-1.5, +-0.5, 63.5 (zeros
    elsewhere): amax 127 -> d = 1, 1/d = 1, codes 127, +-3, +-2, +-1, 64 (half
    away from zero), sum 191 -> s = 191 (binary16 0x59F8; sum h would be
    190.5), d = 1 (0x3C00).  Block 1: h = 63.5, -1.25, 0.75, 0.25, -0.25:
    d = 0.5 (0x3800), 1/d = 2, codes 127, -3, 2, 1, -1, sum 126 -> s = 63
    (0x53E0)."""
    assert oracle.silu32([32.0])[0] == np.float32(32.0)
    K = 64
    g = np.zeros((1, K), np.float32)
    u = np.zeros((1, K), np.float32)
    h0 = [127.0, 2.5, -2.5, 1.5, -1.5, 0.5, -0.5, 63.5]
    pos0 = [3, 5, 6, 10, 11, 20, 21, 31]
    h1 = [63.5, -1.25, 0.75, 0.25, -0.25]
    pos1 = [32 + p for p in (0, 7, 8, 30, 31)]
    for hv, pv in ((h0, pos0), (h1, pos1)):
        for h, p in zip(hv, pv):
            g[0, p] = 32.0
            u[0, p] = h / 32.0
    qs, d, s = oracle.silu_mul_q8_1(g, u)
    want = np.zeros(K, np.int8)
    want[pos0] = [127, 3, -3, 2, -2, 1, -1, 64]
    want[pos1] = [127, -3, 2, 1, -1]
    assert np.array_equal(qs[0], want)
    assert d[0].tolist() == [0x3C00, 0x3800]
    assert s[0].tolist() == [0x59F8, 0x53E0]


def test_silu_mul_q8_1_properties_random():
    """Random gate/up: every block reaches +-127 at its largest |h|, and the
    stored s is fp16(d32 * sum q): within two binary16 roundings of
    d16 * sum q (not the sum of the unquantised products)."""
    B, K = 2, 4096
    g = inputs.activations(17, B, K)
    u = inputs.activations(18, B, K)
    qs, d, s = oracle.silu_mul_q8_1(g, u)
    qb = qs.reshape(B, K // 32, 32).astype(np.int64)
    assert np.all(np.abs(qb).max(-1) == 127)
    ssum = qb.sum(-1).astype(np.float64)
    dd, ss_ = f16(d), f16(s)
    assert np.all(np.abs(ss_ - dd * ssum) <= (2.0 ** -10) * np.abs(dd * ssum) + 1e-7)
    # the dequantised codes approximate h = silu(g) * u within half a step
    gd = g.astype(np.float64)
    h = gd / (1.0 + np.exp(-gd)) * u.astype(np.float64)
    xq = (dd[:, :, None] * qb).reshape(B, K)
    step = np.repeat(dd, 32, axis=1)
    assert np.all(np.abs(xq - h) <= 0.5 * step + 2e-3 * np.abs(h) + 1e-6)
