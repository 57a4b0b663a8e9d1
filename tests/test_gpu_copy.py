"""zq_copy: the SM copy between device memory and mapped pinned host memory.

Byte-exact in every direction, for aligned and unaligned pointers and sizes
with and without a tail past the last 16-byte piece; pointers the device
cannot address are refused before anything runs.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import gemm_zq_rmsnorm_gb300 as zq

pytestmark = pytest.mark.gpu

SIZES = [1, 15, 16, 4103, 135168, 1 << 20]


def _bytes(n, seed):
    return torch.from_numpy(np.random.default_rng(seed).integers(0, 256, n, dtype=np.uint8))


@pytest.mark.parametrize("n", SIZES)
@pytest.mark.parametrize("offset", [0, 1])
def test_copy_host_device_round_trip(n, offset):
    src = _bytes(n + offset, n).pin_memory()[offset:]
    dev = torch.empty(n + offset, dtype=torch.uint8, device="cuda")[offset:]
    back = torch.empty(n + offset, dtype=torch.uint8).pin_memory()[offset:]
    zq.copy(dev, src)                       # pinned host -> device
    torch.cuda.synchronize()
    assert torch.equal(dev.cpu(), src)
    dev2 = torch.empty(n, dtype=torch.uint8, device="cuda")
    zq.copy(dev2, dev)                      # device -> device
    zq.copy(back, dev2)                     # device -> pinned host
    torch.cuda.synchronize()
    assert torch.equal(back, src)
    assert zq.device_status() == 0


def test_copy_ordered_on_stream():
    """A copy reads what the stream's previous kernel wrote, and the next
    kernel sees what the copy wrote."""
    st = torch.cuda.Stream()
    n = 53248
    h = torch.empty(n, dtype=torch.float32).pin_memory()
    with torch.cuda.stream(st):
        x = torch.arange(n, dtype=torch.float32, device="cuda")
        y = x * 3.0
        zq.copy(h, y, stream=st)
        z = torch.empty_like(y)
        zq.copy(z, h, stream=st)
        w = z + 1.0
    st.synchronize()
    assert torch.equal(h, (torch.arange(n, dtype=torch.float32) * 3.0))
    assert torch.equal(w.cpu(), torch.arange(n, dtype=torch.float32) * 3.0 + 1.0)


def test_copy_refuses_pageable_host_memory():
    src = _bytes(256, 1)                    # pageable: not mapped into the device
    dst = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(zq.ZQError):
        zq.copy(dst, src)
    lib = zq.load()
    assert lib.zq_copy(dst.data_ptr(), src.data_ptr(), 0, None) == 0     # nothing to do
    assert lib.zq_copy(None, src.data_ptr(), 16, None) == -1             # ZQ_ERR_ARG
