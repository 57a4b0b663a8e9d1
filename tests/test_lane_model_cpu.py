"""A word-level CPU model of the decode lanes of the streamed mat-vec, checked
against the oracle: the Q4_K in-place high nibbles and byte-permute scale
decoding, the Q5_K fifth bit moved by a funnel rotation, and the Q6_K lane
mapping (2-byte realignment with byte permutes, positions 8p..8p+7 of every
quarter, exact 8-code sums staged in the lanes' order).  It models the
arithmetic of the kernels' lane functions (not the kernels), so edits to those
bit manipulations can be checked without a GPU; the GPU parity tests check the
kernels themselves."""
import struct

import numpy as np

import oracle
from gemm_zq_rmsnorm_gb300 import inputs

M32 = 0xFFFFFFFF


def u32(b, o):
    return struct.unpack_from("<I", bytes(b[o:o + 4]))[0]


def perm(lo, hi, sel):
    """__byte_perm: selector nibbles pick bytes 0..7 of (lo, hi) (3 bits each)."""
    bs = struct.pack("<II", lo, hi)
    return sum(bs[(sel >> (4 * i)) & 7] << (8 * i) for i in range(4))


def rotr(x, r):
    r &= 31
    return ((x >> r) | (x << (32 - r))) & M32 if r else x


def dp4a_us(a, b, c=0):
    """dp4a.u32.s32: unsigned bytes of a times signed bytes of b."""
    for i in range(4):
        bi = (b >> (8 * i)) & 0xFF
        c += ((a >> (8 * i)) & 0xFF) * (bi - 256 if bi > 127 else bi)
    return c


def f16(h):
    return float(np.uint16(h).view(np.float16))


def q8_words(qs, k0, n):
    """n 32-bit words of int8 codes starting at code k0."""
    raw = qs[k0:k0 + 4 * n].astype(np.int8).tobytes()
    return list(struct.unpack("<%dI" % n, raw))


def pair_scales(hdr_words, p):
    """Scales and mins of sub-blocks 2p, 2p+1 from the three scale words."""
    _, y, z, w = hdr_words
    j = (2 * p) & 3
    sel = j | ((j + 1) << 4)
    s0, s1, s2 = perm(y, 0, sel), perm(z, 0, sel), perm(w, 0, sel)
    if p < 2:
        return s0 & 0x3F3F, s1 & 0x3F3F
    return (s2 & 0x0F0F) | ((s0 >> 2) & 0x3030), ((s2 >> 4) & 0x0F0F) | ((s1 >> 2) & 0x3030)


def q45_lane(blk, p, qs, d8, s8, b, five):
    """One lane's part of a Q4_K (five = False) or Q5_K block b of a row."""
    hdr = [u32(blk, 4 * i) for i in range(4)]
    qoff = 48 if five else 16
    ql = [u32(blk, qoff + 32 * p + 4 * k) for k in range(8)]
    a0 = q8_words(qs, 256 * b + 64 * p, 8)          # Q8_1 block 2p
    a1 = q8_words(qs, 256 * b + 64 * p + 32, 8)     # Q8_1 block 2p+1
    if five:
        qh = [u32(blk, 16 + 4 * k) for k in range(8)]
        r0, r1 = (2 * p - 4) & 31, (2 * p - 3) & 31
        I0 = I1 = 0
        for k in range(8):
            q0 = (ql[k] & 0x0F0F0F0F) | (rotr(qh[k], r0) & 0x10101010)
            q1 = ((ql[k] >> 4) & 0x0F0F0F0F) | (rotr(qh[k], r1) & 0x10101010)
            I0, I1 = dp4a_us(q0, a0[k], I0), dp4a_us(q1, a1[k], I1)
    else:
        I0 = I1 = 0
        for k in range(8):
            I0 = dp4a_us(ql[k] & 0x0F0F0F0F, a0[k], I0)
            I1 = dp4a_us(ql[k] & 0xF0F0F0F0, a1[k], I1)   # 16x in place
        assert I1 % 16 == 0
        I1 //= 16
    sc, mn = pair_scales(hdr, p)
    J0, J1 = (sc & 0xFF) * I0, (sc >> 8) * I1
    d, dmin = f16(hdr[0] & 0xFFFF), f16(hdr[0] >> 16)
    c = 8 * b + 2 * p
    main = d8[c + 1] * J1 + d8[c] * J0
    mins = (mn >> 8) * s8[c + 1] + (mn & 0xFF) * s8[c]
    return d * main - dmin * mins


def q6_lane(buf, blk_off, p, qs, d8, b):
    """One lane's part of a Q6_K block at byte blk_off of buf (2-byte aligned)."""
    mis = blk_off & 2
    base4 = blk_off - mis
    sel = 0x5432 if mis else 0x3210

    def ld64(o):
        w0, w1, w2 = (u32(buf, base4 + o + 4 * i) for i in range(3))
        return perm(w0, w1, sel), perm(w1, w2, sel)

    q = [[0, 0] for _ in range(8)]
    for h in range(2):
        hw = ld64(128 + 32 * h + 8 * p)
        for cc in range(2):
            lw = ld64(64 * h + 32 * cc + 8 * p)
            for v in range(2):
                t_lo = (hw[v] << 4 if cc == 0 else hw[v] << 2) & M32
                t_hi = hw[v] if cc == 0 else hw[v] >> 2
                q[4 * h + cc][v] = (lw[v] & 0x0F0F0F0F) | (t_lo & 0x30303030)
                q[4 * h + cc + 2][v] = ((lw[v] >> 4) & 0x0F0F0F0F) | (t_hi & 0x30303030)
    sw = [perm(u32(buf, base4 + 192 + 4 * i), u32(buf, base4 + 196 + 4 * i), sel) for i in range(4)]
    j = p >> 1
    d = f16(struct.unpack_from("<H", bytes(buf[blk_off + 208:blk_off + 210]))[0])
    # the staged 8-code sums in the lanes' order: chunk k8 = 32b + 4q + p
    acc = 0.0
    for qq in range(8):
        a = q8_words(qs, 256 * b + 32 * qq + 8 * p, 2)
        A = int(qs[256 * b + 32 * qq + 8 * p: 256 * b + 32 * qq + 8 * p + 8].astype(np.int64).sum())
        I = dp4a_us(q[qq][1], a[1], dp4a_us(q[qq][0], a[0])) - 32 * A
        sb = (sw[qq >> 1] >> (8 * (j + 2 * (qq & 1)))) & 0xFF
        sc = sb - 256 if sb > 127 else sb
        acc += float(d8[8 * b + qq]) * (sc * I)
    return d * acc


def _q8(seed, K):
    x = inputs.activations(seed, 1, K)
    qs, d, s = oracle.rmsnorm_q8_1(x, inputs.gamma(seed, K), inputs.EPS)
    return qs[0], d, s, f16_arr(d[0]), f16_arr(s[0])


def f16_arr(h):
    return np.asarray(h, np.uint16).view(np.float16).astype(np.float64)


def test_q4k_and_q5k_lane_model():
    K, N = 512, 6
    qs, d, s, d8, s8 = _q8(3, K)
    for five, gen in ((False, inputs.q4k_weights), (True, inputs.q5k_weights)):
        W = gen(3, N, K)
        kb = 176 if five else 144
        y_ref, S = oracle.kq_matmul("q5k" if five else "q4k", W, N, K, qs[None], d, s)
        for n in range(N):
            y = 0.0
            for b in range(K // 256):
                blk = W[n, b * kb:(b + 1) * kb]
                y += sum(q45_lane(blk, p, qs, d8, s8, b, five) for p in range(4))
            assert abs(y - y_ref[0, n]) <= 1e-9 * S[0, n] + 1e-7 * abs(y_ref[0, n]), (five, n)


def test_q6k_lane_model_both_alignments():
    K, N = 512, 5
    qs, d, s, d8, _ = _q8(4, K)
    W = inputs.q6k_weights(4, N, K)
    y_ref, S = oracle.kq_matmul("q6k", W, N, K, qs[None], d, s)
    for shift in (0, 2, 6):                      # block start mod 4 = 0 and 2
        buf = bytearray(W.size + 16)
        buf[shift:shift + W.size] = W.tobytes()
        for n in range(N):
            y = 0.0
            for b in range(K // 256):
                off = shift + (n * (K // 256) + b) * 210
                y += sum(q6_lane(buf, off, p, qs, d8, b) for p in range(4))
            assert abs(y - y_ref[0, n]) <= 1e-9 * S[0, n] + 1e-7 * abs(y_ref[0, n]), (shift, n)


def test_funnel_rotation_moves_each_bit_within_its_byte():
    rng = np.random.default_rng(0)
    for p in range(4):
        for j, r in ((2 * p, (2 * p - 4) & 31), (2 * p + 1, (2 * p - 3) & 31)):
            for qh in rng.integers(0, 2 ** 32, 500, dtype=np.uint64):
                qh = int(qh)
                want = sum(1 << (8 * i + 4) for i in range(4) if (qh >> (8 * i + j)) & 1)
                assert rotr(qh, r) & 0x10101010 == want
