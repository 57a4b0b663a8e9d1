"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module holds no step of the method's arithmetic (no normalisation, no
quantisation of activations, no dot products).  It draws random numbers and
lays them out in the storage formats the library reads:

* activations x: fp32 N(0,1) (Box-Muller in fp64, rounded to fp32), with 1 %
  of the feature channels (the same channels for every token) scaled by 20;
* gamma: fp32 U(0.5, 1.5);
* Q4_K weights: per 256-weight super-block, quants U{0..15}, 6-bit scales
  U{1..63}, 6-bit mins U{0..63}, d and dmin = binary16(U(1e-4, 1e-3)),
  packed into the 144-byte block layout (d, dmin, 12 scale bytes, 128 nibble
  bytes) that the library's header documents.

All randomness comes from splitmix64 used as a counter-based generator:
value i of a stream with key k is mix(k + (i+1)*0x9E3779B97F4A7C15), where
mix is the splitmix64 output function; each tensor gets its own key derived
from the seed and a fixed tag, so streams are independent and every tensor
is reproducible on its own on any machine.
"""
from __future__ import annotations

import dataclasses

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# fixed stream tags
TAG_X, TAG_GAMMA, TAG_OUTLIER = 1, 2, 3
TAG_Q, TAG_SC, TAG_M, TAG_D, TAG_DMIN = 10, 11, 12, 13, 14


def _mix(z: np.ndarray) -> np.ndarray:
    z = z.astype(np.uint64, copy=True)
    z ^= z >> np.uint64(30)
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def stream_key(seed: int, tag: int) -> np.uint64:
    with np.errstate(over="ignore"):
        base = np.array([np.uint64(seed & 0xFFFFFFFFFFFFFFFF)], np.uint64) * _GOLDEN
        return _mix(base + np.uint64(tag))[0]


def bits(seed: int, tag: int, n: int, offset: int = 0) -> np.ndarray:
    """n raw 64-bit values of stream (seed, tag), starting at counter offset."""
    key = stream_key(seed, tag)
    with np.errstate(over="ignore"):
        ctr = np.arange(offset + 1, offset + n + 1, dtype=np.uint64)
        return _mix(key + ctr * _GOLDEN)


def uniform01(seed: int, tag: int, n: int) -> np.ndarray:
    """fp64 uniforms in [0, 1) from the top 53 bits."""
    return (bits(seed, tag, n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal(seed: int, tag: int, n: int) -> np.ndarray:
    """fp64 N(0,1) by Box-Muller (cosine branch), two uniforms per value."""
    u = uniform01(seed, tag, 2 * n).reshape(n, 2)
    return np.sqrt(-2.0 * np.log1p(-u[:, 0])) * np.cos(2.0 * np.pi * u[:, 1])


def uniform_int(seed: int, tag: int, n: int, lo: int, hi: int) -> np.ndarray:
    """Integers uniform on [lo, hi] (inclusive) via the multiply-high map."""
    span = hi - lo + 1
    top = (bits(seed, tag, n) >> np.uint64(32)).astype(np.uint64)  # 32 bits
    return (lo + ((top * np.uint64(span)) >> np.uint64(32))).astype(np.int64)


# --------------------------------------------------------------------------
# activations
# --------------------------------------------------------------------------
def outlier_channels(seed: int, K: int, frac: float = 0.01) -> np.ndarray:
    """round(frac*K) distinct feature indices, a seeded random subset."""
    n = int(round(frac * K))
    keys = bits(seed, TAG_OUTLIER, K)
    return np.sort(np.argsort(keys, kind="stable")[:n])


def activations(seed: int, B: int, K: int, outlier_scale: float = 20.0) -> np.ndarray:
    """x fp32 [B][K]: N(0,1), the outlier channels scaled by outlier_scale."""
    x = normal(seed, TAG_X, B * K).reshape(B, K)
    ch = outlier_channels(seed, K)
    x[:, ch] *= outlier_scale
    return x.astype(np.float32)


def gamma(seed: int, K: int) -> np.ndarray:
    return (0.5 + uniform01(seed, TAG_GAMMA, K)).astype(np.float32)


# --------------------------------------------------------------------------
# Q4_K weights
# --------------------------------------------------------------------------
@dataclasses.dataclass
class Q4KFields:
    """Unpacked fields of an N x K Q4_K matrix (nb = K/256 super-blocks/row)."""
    d: np.ndarray      # uint16 binary16 bits [N, nb]
    dmin: np.ndarray   # uint16 binary16 bits [N, nb]
    sc: np.ndarray     # uint8 [N, nb, 8], 0..63
    m: np.ndarray      # uint8 [N, nb, 8], 0..63
    q: np.ndarray      # uint8 [N, nb, 8, 32], 0..15


def q4k_fields(seed: int, N: int, K: int, *, tag_offset: int = 0) -> Q4KFields:
    assert K % 256 == 0 and K > 0 and N > 0
    nb = K // 256
    nblk = N * nb
    raw = bits(seed, TAG_Q + tag_offset, nblk * 16)  # 16 nibbles per uint64
    shifts = (np.arange(16, dtype=np.uint64) * np.uint64(4))
    q = ((raw[:, None] >> shifts[None, :]) & np.uint64(15)).astype(np.uint8)
    q = q.reshape(N, nb, 8, 32)
    sc = uniform_int(seed, TAG_SC + tag_offset, nblk * 8, 1, 63).astype(np.uint8).reshape(N, nb, 8)
    m = uniform_int(seed, TAG_M + tag_offset, nblk * 8, 0, 63).astype(np.uint8).reshape(N, nb, 8)
    dv = 1e-4 + 9e-4 * uniform01(seed, TAG_D + tag_offset, nblk)
    dmv = 1e-4 + 9e-4 * uniform01(seed, TAG_DMIN + tag_offset, nblk)
    d = dv.astype(np.float16).view(np.uint16).reshape(N, nb)
    dmin = dmv.astype(np.float16).view(np.uint16).reshape(N, nb)
    return Q4KFields(d=d, dmin=dmin, sc=sc, m=m, q=q)


def pack_q4k(f: Q4KFields) -> np.ndarray:
    """Encode fields into the 144-byte block layout; returns uint8 [N, nb*144].

    bytes 0..1 d, 2..3 dmin (little-endian binary16); bytes 4..15 scales S:
      S[j]   = sc[j] | (sc[j+4] >> 4) << 6        (j = 0..3)
      S[j+4] = m[j]  | (m[j+4]  >> 4) << 6        (j = 0..3)
      S[j+8] = (sc[j+4] & 15) | (m[j+4] & 15) << 4 (j = 0..3)
    bytes 16..143: byte 32*p + i = q[2p][i] | q[2p+1][i] << 4 (p = 0..3).
    """
    N, nb = f.d.shape
    assert f.sc.max() < 64 and f.m.max() < 64 and f.q.max() < 16
    out = np.zeros((N, nb, 144), np.uint8)
    out[:, :, 0] = (f.d & 0xFF).astype(np.uint8)
    out[:, :, 1] = (f.d >> 8).astype(np.uint8)
    out[:, :, 2] = (f.dmin & 0xFF).astype(np.uint8)
    out[:, :, 3] = (f.dmin >> 8).astype(np.uint8)
    sc = f.sc.astype(np.uint16)
    m = f.m.astype(np.uint16)
    S = np.zeros((N, nb, 12), np.uint16)
    S[:, :, 0:4] = sc[:, :, 0:4] | ((sc[:, :, 4:8] >> 4) << 6)
    S[:, :, 4:8] = m[:, :, 0:4] | ((m[:, :, 4:8] >> 4) << 6)
    S[:, :, 8:12] = (sc[:, :, 4:8] & 15) | ((m[:, :, 4:8] & 15) << 4)
    out[:, :, 4:16] = S.astype(np.uint8)
    q = f.q.astype(np.uint8)
    nib = q[:, :, 0::2, :] | (q[:, :, 1::2, :] << 4)  # [N, nb, 4, 32]
    out[:, :, 16:144] = nib.reshape(N, nb, 128)
    return out.reshape(N, nb * 144)


def q4k_weights(seed: int, N: int, K: int, *, tag_offset: int = 0) -> np.ndarray:
    return pack_q4k(q4k_fields(seed, N, K, tag_offset=tag_offset))


# --------------------------------------------------------------------------
# Q5_K and Q6_K weights (the other k-quant blocks of Q4_K_M checkpoints)
# --------------------------------------------------------------------------
TAG_QH, TAG_Q6, TAG_Q6SC, TAG_Q6D = 15, 16, 17, 18


@dataclasses.dataclass
class Q5KFields:
    """Unpacked fields of an N x K Q5_K matrix: as Q4_K, with 5-bit quants."""
    d: np.ndarray      # uint16 binary16 bits [N, nb]
    dmin: np.ndarray   # uint16 binary16 bits [N, nb]
    sc: np.ndarray     # uint8 [N, nb, 8], 0..63
    m: np.ndarray      # uint8 [N, nb, 8], 0..63
    q: np.ndarray      # uint8 [N, nb, 8, 32], 0..31


def q5k_fields(seed: int, N: int, K: int, *, tag_offset: int = 0) -> Q5KFields:
    """Scales, mins and d/dmin drawn as for Q4_K; quants U{0..31} (the low
    four bits from the Q4_K nibble stream, the fifth from a stream of its own)."""
    f4 = q4k_fields(seed, N, K, tag_offset=tag_offset)
    nblk = N * (K // 256)
    raw = bits(seed, TAG_QH + tag_offset, nblk * 4)            # 64 high bits per uint64
    shifts = np.arange(64, dtype=np.uint64)
    hb = ((raw[:, None] >> shifts[None, :]) & np.uint64(1)).astype(np.uint8)
    q = f4.q | (hb.reshape(f4.q.shape) << 4)
    return Q5KFields(d=f4.d, dmin=f4.dmin, sc=f4.sc, m=f4.m, q=q)


def pack_q5k(f: Q5KFields) -> np.ndarray:
    """Encode fields into the 176-byte block layout; returns uint8 [N, nb*176].

    bytes 0..15 as Q4_K (d, dmin, the twelve scale/min bytes);
    bytes 16..47 qh: bit j of byte 16+i = bit 4 of q[j][i];
    bytes 48..175: byte 48 + 32*p + i = (q[2p][i] & 15) | (q[2p+1][i] & 15) << 4.
    """
    N, nb = f.d.shape
    assert f.q.max() < 32
    low = pack_q4k(Q4KFields(d=f.d, dmin=f.dmin, sc=f.sc, m=f.m, q=f.q & 15)).reshape(N, nb, 144)
    out = np.zeros((N, nb, 176), np.uint8)
    out[:, :, 0:16] = low[:, :, 0:16]
    hb = (f.q >> 4).astype(np.uint16)                           # [N, nb, 8, 32]
    qh = np.zeros((N, nb, 32), np.uint16)
    for j in range(8):
        qh |= hb[:, :, j, :] << j
    out[:, :, 16:48] = qh.astype(np.uint8)
    out[:, :, 48:176] = low[:, :, 16:144]
    return out.reshape(N, nb * 176)


def q5k_weights(seed: int, N: int, K: int, *, tag_offset: int = 0) -> np.ndarray:
    return pack_q5k(q5k_fields(seed, N, K, tag_offset=tag_offset))


@dataclasses.dataclass
class Q6KFields:
    """Unpacked fields of an N x K Q6_K matrix (16 sub-blocks of 16 weights)."""
    d: np.ndarray      # uint16 binary16 bits [N, nb]
    sc: np.ndarray     # int8 [N, nb, 16], -128..127
    q: np.ndarray      # uint8 [N, nb, 16, 16], 0..63 (weight value d*sc*(q-32))


def q6k_fields(seed: int, N: int, K: int, *, tag_offset: int = 0) -> Q6KFields:
    """Quants U{0..63}, scales U{-128..127} (the full int8 range), d =
    binary16(U(1e-5, 1e-4)) so that |d*sc*(q-32)| stays below 0.41 like the
    Q4_K weights."""
    assert K % 256 == 0 and K > 0 and N > 0
    nb = K // 256
    nblk = N * nb
    raw = bits(seed, TAG_Q6 + tag_offset, nblk * 32)            # 8 six-bit quants per uint64
    shifts = np.arange(8, dtype=np.uint64) * np.uint64(6)
    q = ((raw[:, None] >> shifts[None, :]) & np.uint64(63)).astype(np.uint8).reshape(N, nb, 16, 16)
    sc = (uniform_int(seed, TAG_Q6SC + tag_offset, nblk * 16, 0, 255) - 128).astype(np.int8).reshape(N, nb, 16)
    dv = 1e-5 + 9e-5 * uniform01(seed, TAG_Q6D + tag_offset, nblk)
    d = dv.astype(np.float16).view(np.uint16).reshape(N, nb)
    return Q6KFields(d=d, sc=sc, q=q)


def pack_q6k(f: Q6KFields) -> np.ndarray:
    """Encode fields into the 210-byte block layout; returns uint8 [N, nb*210].

    Weight k (0..255) of a block has half h = k // 128, and within the half
    quarter c = (k % 128) // 32 and position i = k % 32:
      low four bits of q in byte 64*h + 32*(c % 2) + i (bytes 0..127), low
        nibble for c < 2, high nibble for c >= 2;
      top two bits of q in bits 2c, 2c+1 of byte 128 + 32*h + i (bytes 128..191);
    bytes 192..207: the 16 int8 scales, sc[s] for weights 16s..16s+15;
    bytes 208..209: d (little-endian binary16).
    """
    N, nb = f.d.shape
    assert f.q.max() < 64
    q = f.q.reshape(N, nb, 2, 4, 32).astype(np.uint16)          # [.., h, c, i]
    out = np.zeros((N, nb, 210), np.uint8)
    lo = q & 15
    ql = np.zeros((N, nb, 2, 2, 32), np.uint16)                 # [.., h, c % 2, i]
    ql[:, :, :, 0, :] = lo[:, :, :, 0, :] | (lo[:, :, :, 2, :] << 4)
    ql[:, :, :, 1, :] = lo[:, :, :, 1, :] | (lo[:, :, :, 3, :] << 4)
    out[:, :, 0:128] = ql.reshape(N, nb, 128).astype(np.uint8)
    hi = q >> 4
    qh = np.zeros((N, nb, 2, 32), np.uint16)
    for c in range(4):
        qh |= hi[:, :, :, c, :] << (2 * c)
    out[:, :, 128:192] = qh.reshape(N, nb, 64).astype(np.uint8)
    out[:, :, 192:208] = f.sc.view(np.uint8)
    out[:, :, 208] = (f.d & 0xFF).astype(np.uint8)
    out[:, :, 209] = (f.d >> 8).astype(np.uint8)
    return out.reshape(N, nb * 210)


def q6k_weights(seed: int, N: int, K: int, *, tag_offset: int = 0) -> np.ndarray:
    return pack_q6k(q6k_fields(seed, N, K, tag_offset=tag_offset))


# --------------------------------------------------------------------------
# named workloads (shapes of the pages' models; every input synthetic)
# --------------------------------------------------------------------------
EPS = 1e-6

# (name, K, N, paired) ; paired = gate/up run as one pair kernel
TINY = [("proj", 1024, 1024, False)]
SMALL_DECODE = [  # hidden 1024, 28-ish-layer small model, plus the LM head
    ("q_proj", 1024, 2048, False), ("k_proj", 1024, 1024, False),
    ("v_proj", 1024, 1024, False), ("o_proj", 2048, 1024, False),
    ("gate_up", 1024, 3072, True), ("down", 3072, 1024, False),
    ("lm_head", 1024, 151936, False)]
LAYER_27B = [  # one decoder layer of a 27B-class model, hidden 5120
    ("q_proj", 5120, 6144, False), ("k_proj", 5120, 1024, False),
    ("v_proj", 5120, 1024, False), ("o_proj", 6144, 5120, False),
    ("gate_up", 5120, 17408, True), ("down", 17408, 5120, False)]
CHUNK_SHAPES = [("down", 17408, 5120, False), ("gate_up", 5120, 17408, True)]
CHUNK_BATCHES = (4, 8, 16)
PREFILL_B = 512
