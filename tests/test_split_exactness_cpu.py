"""The batched projection's activation split (q8_split_kernel): each Q8_1 value
x' = q8 * d8 is written as two binary16 numbers hi = fp16(x') and
lo = fp16(x' - hi).  Checked exhaustively here, for every finite binary16 scale
d8 with 127 * d8 within binary16 range and every code q8 in [-127, 127]: x' is
exact in fp32, x' - hi is exact in fp32, lo is exactly representable, so
hi + lo == x' and every product of hi or lo with a weight code sc*q4 (<= 945,
exact in binary16) is exact in the fp32 accumulation."""
import numpy as np


def test_hi_lo_split_is_exact_for_every_scale_and_code():
    h = np.arange(0x0001, 0x7C00, dtype=np.uint32).astype(np.uint16)   # positive finite binary16
    d8 = h.view(np.float16).astype(np.float32)
    d8 = d8[127.0 * d8.astype(np.float64) <= 65504.0]                  # tokens that need no 2^-k scaling
    q8 = np.arange(-127, 128, dtype=np.float32)
    x = (q8[None, :] * d8[:, None]).astype(np.float32)                 # fp32 product, as the kernel forms it
    exact = q8[None, :].astype(np.float64) * d8[:, None].astype(np.float64)
    assert np.array_equal(x.astype(np.float64), exact)                 # 7 x 11 bits fit in 24
    hi = x.astype(np.float16)
    rem = (x - hi.astype(np.float32)).astype(np.float32)
    assert np.array_equal(rem.astype(np.float64), x.astype(np.float64) - hi.astype(np.float64))
    lo = rem.astype(np.float16)
    assert np.array_equal(lo.astype(np.float64), rem.astype(np.float64))   # lo exact in binary16
    assert np.array_equal(hi.astype(np.float64) + lo.astype(np.float64), exact)
    # products with the largest weight code stay exact in fp32 (<= 24 significant bits)
    for part in (hi, lo):
        p = part.astype(np.float64) * 945.0
        assert np.array_equal(p.astype(np.float32).astype(np.float64), p)


def test_nibble_to_binary16_fma_is_exact():
    """The converter warps turn a nibble q and a 6-bit scale s into s*q with one
    binary16 fma: low nibble in the mantissa of 1024 (h = 1024 + q), scale s,
    offset -1024 s; high nibble in place (h = 1024 + 16 q), scale s/16, offset
    -64 s.  Every operand is exact in binary16 and the one rounding of the fma
    meets an exactly representable result (s*q <= 945 < 2048)."""
    for s in range(64):
        for q in range(16):
            for h, scale, off in ((1024 + q, s, -1024 * s), (1024 + 16 * q, s / 16, -64 * s)):
                for v in (h, scale, off):
                    assert float(np.float16(v)) == v          # operands exact in binary16
                fused = np.float16(h * scale + off)            # one rounding of the exact value
                assert float(fused) == s * q
