"""Bit-exact projections on inputs whose fp32 arithmetic is exact.

The tolerance tests allow |err| <= 1e-4 * S, so a kernel mistake that adds a
small error (a dropped low half of the split activations, a mis-scaled min
product, one sub-block's scale applied to its neighbour at the 1e-5 level)
could pass them.  Here every quantity is a small integer times a power of two:

* d = dmin = 2^-10 for every super-block;
* token t's Q8_1 scales are d8 = m8 * 2^e_t with m8 in 16..31 (five bits), so
  a value q8 * d8 with |q8| >= 67 has twelve significant bits and its binary16
  split has a non-zero low half;
* the block sums s8 are m8 * r * 2^e_t with |m8 * r| < 2048 (exact in
  binary16; the projection takes the s plane as given).

Every product and every partial sum of y[t][n] is then an integer multiple of
2^(e_t - 10); the fixture asserts that the sum of the absolute values of all
terms of every output stays below 2^23 such units, so any fp32 summation
order is exact, and the oracle's fp64 result rounds to the same fp32 value.
The GPU result must equal the oracle bit for bit, through zq_q4k_gemm at
every batch-size branch: B = 1 (decode mat-vec), 4 (streamed tokens), 5..16
(small-batch tensor-core kernel), 130 and 512 (128-token tiles), with split-K
and a ragged N.  One token per batch uses e_t = 5, which makes 127 * max d8
exceed the binary16 range, so the power-of-two token scaling runs too.

Two weight/activation mixes keep the bound: "dense" (all codes in -127..127,
weights sc * q4 with q4 in {0, 1}, sc in {1, 2}, mins in {0, 1}) and "sparse"
(two non-zero codes per token, full-range quants, scales and mins).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import gemm_zq_rmsnorm_gb300 as zq
from gemm_zq_rmsnorm_gb300 import inputs

pytestmark = pytest.mark.gpu

F16_2M10 = 0x1400            # binary16 of 2^-10


def _exact_case(seed, B, K, N, mix):
    nb, nblk = K // 256, K // 32
    f = inputs.q4k_fields(seed, N, K)
    f.d[...] = F16_2M10
    f.dmin[...] = F16_2M10
    if mix == "dense":
        f.q[...] = (f.q & 1).astype(np.uint8)
        f.sc[...] = (1 + (f.sc & 1)).astype(np.uint8)
        f.m[...] = (f.m & 1).astype(np.uint8)
        qs = (inputs.uniform_int(seed, 901, B * K, 0, 254) - 127).reshape(B, K).astype(np.int8)
        rmax = 60
    else:
        qs = np.zeros((B, K), np.int8)
        pos = inputs.uniform_int(seed, 902, 2 * B, 0, K - 1).reshape(B, 2)
        mag = inputs.uniform_int(seed, 903, 2 * B, 67, 127).reshape(B, 2)
        sgn = np.where(inputs.uniform_int(seed, 904, 2 * B, 0, 1).reshape(B, 2) == 1, 1, -1)
        for t in range(B):
            for c in range(2):
                qs[t, pos[t, c]] = mag[t, c] * sgn[t, c]
        rmax = 15 if K > 2048 else 30
    m8 = inputs.uniform_int(seed, 905, B * nblk, 16, 31).reshape(B, nblk).astype(np.int64)
    if mix == "sparse":
        # the first code of every token: odd, >= 67, in a block with m8 = 31,
        # so q8 * m8 is odd with twelve bits and its low binary16 half is non-zero
        for t in range(B):
            qs[t, pos[t, 0]] = (67 + 2 * (mag[t, 0] % 31)) * sgn[t, 0]
            m8[t, pos[t, 0] // 32] = 31
    r = (inputs.uniform_int(seed, 906, B * nblk, 0, 2 * rmax) - rmax).reshape(B, nblk).astype(np.int64)
    e = np.full(B, -9, np.int64)
    e[B // 2] = 5                                        # 127 * 31 * 2^5 > 65504: token scaling
    d8 = (m8 * np.exp2(e)[:, None]).astype(np.float16)
    s8 = (m8 * r * np.exp2(e)[:, None]).astype(np.float16)
    assert np.array_equal(d8.astype(np.float64), m8 * np.exp2(e)[:, None])
    assert np.array_equal(s8.astype(np.float64), m8 * r * np.exp2(e)[:, None])
    W = inputs.pack_q4k(f)
    # the exactness bound, in integer units of 2^(e_t - 10)
    w = (f.sc[:, :, :, None].astype(np.int64) * f.q).reshape(N, K)
    xq = qs.astype(np.int64) * np.repeat(m8, 32, axis=1)            # q8 * d8 / 2^e_t
    main = np.abs(xq) @ np.abs(w).T                                 # [B][N]
    mins = np.abs(m8 * r) @ f.m.reshape(N, nblk).T.astype(np.int64)
    assert (main + mins).max() < 2 ** 23, "fixture outside the exact range"
    lo_nonzero = np.count_nonzero((np.abs(xq) >= 2048) & (xq % 2 != 0))   # 12 significant bits
    return W, qs, d8.view(np.uint16), s8.view(np.uint16), lo_nonzero


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda")


@pytest.mark.parametrize("mix", ["dense", "sparse"])
@pytest.mark.parametrize("B,K,N", [(1, 1280, 200), (4, 1280, 200), (5, 1280, 200), (8, 1280, 200),
                                   (16, 1280, 200), (130, 1280, 200), (512, 1280, 200), (16, 5120, 136),
                                   (512, 5120, 136)])
def test_projection_bit_exact_when_arithmetic_is_exact(mix, B, K, N):
    if mix == "dense" and K > 2048:
        pytest.skip("the dense mix stays exact up to K = 2048")
    W, qs, d, s, lo_nonzero = _exact_case(300 + B + K, B, K, N, mix)
    assert lo_nonzero > 0                     # some values need both binary16 halves
    a = zq.Q8_1(_dev(qs), _dev(d.view(np.float16)), _dev(s.view(np.float16)))
    y = zq.q4k_gemm(_dev(W), N, K, a, B)
    torch.cuda.synchronize()
    assert zq.device_status() == 0
    got = y.cpu().numpy().reshape(B, N)
    ref, _ = oracle.q4k_matmul(W, N, K, qs, d, s)
    ref = ref.astype(np.float32)
    bad = got.view(np.uint32) != ref.view(np.uint32)
    assert not bad.any(), (f"{bad.sum()} outputs differ, first {np.argwhere(bad)[:3].tolist()}: "
                           f"gpu {got[bad][:3]} oracle {ref[bad][:3]}")
