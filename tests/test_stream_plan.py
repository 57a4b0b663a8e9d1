"""CPU checks of the streamed mat-vec's launch plan (the host code the kernel
launches with, through the zq_debug_stream_plan hook): shared memory within
the per-CTA limit, every stage large enough for its tile and, for Q6_K, for
the 16-byte-aligned copy around it, reductions within their bounds, and a
row's summation order (pieces and segments) fixed by K alone."""
import os

import pytest

import gemm_zq_rmsnorm_gb300 as zq
from gemm_zq_rmsnorm_gb300 import build as zqbuild

BLOCK = {4: 144, 5: 176, 6: 210}
SMEM_LIMIT = 227 * 1024 - 1024           # dynamic bytes (static shared memory pads to 1 KB)
MAX_TASKS = 65536 // 144                 # contribution slots per stage
KS = [256, 512, 768, 1024, 1536, 2048, 2816, 3072, 4096, 5120, 6144, 8192, 12288, 17408, 20480, 29696, 32768]


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not os.path.exists(zq.LIB_PATH):
        zqbuild.build()
    return zq.load()


def plan(fmt, nt, K, rows, sms=152):
    return zq.debug_stream_plan(fmt, nt, K, rows, sms)


def fits(fmt, nt, K):
    try:
        plan(fmt, nt, K, 1000)
        return True
    except zq.ZQError as e:
        assert e.status == -2
        return False


@pytest.mark.parametrize("fmt", [4, 5, 6])
@pytest.mark.parametrize("nt", [1, 4])
def test_plan_invariants(fmt, nt):
    kb = BLOCK[fmt]
    slack = 32 if kb % 16 else 0
    for K in KS:
        if not fits(fmt, nt, K):
            assert nt == 4 and fmt == 6 and K > 29696
            continue
        nb = K // 256
        shapes = []
        for rows in (1, 7, 300, 5120, 34816, 151936):
            for sms in (148, 152):
                p = plan(fmt, nt, K, rows, sms)
                assert p["rowbytes"] == nb * kb
                assert p["smem"] <= SMEM_LIMIT, (K, rows, p)
                assert p["stage_alloc"] % 128 == 0
                if p["P"] == 1:
                    assert p["CB"] == nb and p["R"] >= 1
                    assert p["stage_alloc"] >= p["R"] * p["rowbytes"] + slack
                else:
                    assert p["R"] == 1 and p["CB"] * (p["P"] - 1) < nb <= p["CB"] * p["P"]
                    assert p["stage_alloc"] >= p["CB"] * kb + slack
                if p["wl"]:
                    assert p["P"] == 1 and p["nseg"] in (1, 2, 4, 8)
                else:
                    blocks = nb if p["P"] == 1 else p["CB"]
                    assert p["nseg"] <= 32                        # one lane per segment in the row reduction
                    assert p["R"] * p["nseg"] <= MAX_TASKS or p["P"] > 1
                    assert -(-blocks // p["nseg"]) <= 4 or p["nseg"] == blocks
                shapes.append((p["P"], p["CB"], p["nseg"], p["wl"]))
        # a row's summation order does not depend on the other rows of the launch
        assert len(set(shapes)) == 1, (fmt, nt, K, set(shapes))


def test_q6k_four_token_limit():
    assert fits(6, 4, 29696) and not fits(6, 4, 29952)
    assert fits(4, 4, 32768) and fits(5, 4, 32768)


@pytest.mark.parametrize("K", [256, 1024, 5120, 17408, 32768])
@pytest.mark.parametrize("N", [1, 7, 61, 300])
def test_q6k_aligned_copies_stay_in_the_stage_and_the_buffer(K, N):
    """The producer copies [start rounded down to 16, end rounded up to 16),
    clipped at the matrix's last 16-byte boundary (the rest by plain loads):
    every copy must fit the stage, start inside the matrix and end inside it."""
    p = plan(6, 1, K, N)
    rb, total = p["rowbytes"], N * p["rowbytes"]
    nb = K // 256
    for g in range(-(-N // p["R"])):
        row0 = g * p["R"]
        rows = min(p["R"], N - row0)
        for pc in range(p["P"]):
            nbytes = rows * rb if p["P"] == 1 else min(p["CB"], nb - pc * p["CB"]) * 210
            start = row0 * rb + pc * p["CB"] * 210
            end = start + nbytes
            lo = start & ~15
            hi = min((end + 15) & ~15, total & ~15)
            assert 0 <= lo < hi <= total and (hi - lo) % 16 == 0
            assert end - hi < 16                              # the plain-load tail
            assert hi - lo <= p["stage_alloc"]
            assert (start & 15) + nbytes + 2 <= p["stage_alloc"]   # last block's aligned reads
