"""Failure path of the bounded waits, on the GPU, without a fault.

The streamed mat-vec is launched through its test hook with a short wait limit
and a producer that stops before issuing one stage.  No copy is then in
flight; the consumers' wait for the withheld stage must run out, every role of
the kernel must return, the device status word must carry bit 0, and the rows
of the stages before the withheld one must still be right.  Afterwards the
same context must run an ordinary projection correctly.
"""
import time

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import gemm_zq_rmsnorm_gb300 as zq

from _cases import assert_within, make_layer_inputs, oracle_q8

pytestmark = pytest.mark.gpu

DEV = "cuda"
WAIT_US = 1000


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def q8_dev(qs, d, s) -> zq.Q8_1:
    return zq.Q8_1(to_dev(qs), to_dev(d.view(np.float16)), to_dev(s.view(np.float16)))


def plan(K, N, ctas):
    p = zq.debug_stream_plan(4, 1, K, N, ctas)
    return p["R"], p["P"], p["wl"]


@pytest.mark.parametrize("K,N,ctas,withhold", [
    (2560, 64, 1, 1),      # warp-local rows; stage 0 runs, stage 1 withheld
    (32768, 16, 1, 1),     # rows reduced through shared memory
    (2560, 64, 1, 2),
    (1024, 600, 4, 0),     # nothing issued at all, four CTAs
])
def test_wait_expires_and_reports(K, N, ctas, withhold):
    x, g, W = make_layer_inputs(900 + K + N, 1, K, N)
    qs, d, s = oracle_q8(x, g)
    y_ref, S = oracle.q4k_matmul(W, N, K, qs, d, s)
    R, P, wl = plan(K, N, ctas)
    assert P == 1
    groups = (N + R - 1) // R
    # CTA c handles groups c, c + ctas, ...: its stage j is group c + j * ctas
    assert groups > withhold * ctas, "every CTA must have a stage to withhold"

    assert zq.device_status(clear=True) == 0
    Wd, a = to_dev(W), q8_dev(qs, d, s)
    y = torch.full((N,), float("nan"), dtype=torch.float32, device=DEV)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    zq.debug_wait_expiry(Wd, N, K, a, y, withhold, WAIT_US, ctas)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert zq.device_status(clear=True) == zq.DEVICE_WAIT_EXPIRED
    # the short limit, not the two-second default, ended the waits
    assert elapsed < 0.5, elapsed

    got = y.cpu().numpy()
    done = np.zeros(N, bool)
    for c in range(ctas):
        for j in range(withhold):
            grp = c + j * ctas
            if grp < groups:
                done[grp * R:min(N, (grp + 1) * R)] = True
    if done.any():
        assert_within(got[None, done], y_ref[:, done], S[:, done], "stages before the withheld one")
    assert np.all(np.isnan(got[~done])), "rows of withheld stages were written"

    # the context is healthy: an ordinary launch is right and raises nothing
    y2 = zq.q4k_gemv(Wd, N, K, a)
    torch.cuda.synchronize()
    assert zq.device_status() == 0
    assert_within(y2.cpu().numpy()[None], y_ref, S, "after expiry")


def test_withhold_past_the_work_changes_nothing():
    """A withheld stage the CTAs never reach: no wait expires, every row is right."""
    K, N = 2560, 64
    x, g, W = make_layer_inputs(950, 1, K, N)
    qs, d, s = oracle_q8(x, g)
    y_ref, S = oracle.q4k_matmul(W, N, K, qs, d, s)
    assert zq.device_status(clear=True) == 0
    y = torch.full((N,), float("nan"), dtype=torch.float32, device=DEV)
    zq.debug_wait_expiry(to_dev(W), N, K, q8_dev(qs, d, s), y, 1000, WAIT_US, 1)
    torch.cuda.synchronize()
    assert zq.device_status() == 0
    assert_within(y.cpu().numpy()[None], y_ref, S, "withhold past the work")


def test_wait_expiry_argument_checks():
    K, N = 256, 8
    W = torch.zeros(zq.q4k_bytes(N, K), dtype=torch.uint8, device=DEV)
    a = zq.Q8_1(torch.zeros(K, dtype=torch.int8, device=DEV), torch.zeros(K // 32, dtype=torch.float16, device=DEV),
                torch.zeros(K // 32, dtype=torch.float16, device=DEV))
    y = torch.empty(N, dtype=torch.float32, device=DEV)
    for withhold, wait_us, ctas in ((-1, 1000, 1), (0, 0, 1), (0, 3_000_000, 1), (0, 1000, 0), (0, 1000, 100000)):
        with pytest.raises(zq.ZQError):
            zq.debug_wait_expiry(W, N, K, a, y, withhold, wait_us, ctas)
    assert zq.device_status() == 0
