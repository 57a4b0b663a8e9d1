"""The toolchain facts the batched projection's design rests on, checked
with the installed nvcc (no GPU needed): the int8 tcgen05 MMA
(`tcgen05.mma ... .kind::i8`) is rejected for sm_103a, so the prefill path
runs binary16 MMAs; the same instruction assembles for sm_100a, so the
rejection is about the target, not the syntax."""
import os
import shutil
import subprocess
import tempfile

import pytest

NVCC = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"

SRC = r'''
#include <stdint.h>
__global__ void k(uint32_t d, uint64_t a, uint64_t b, uint32_t i, int *o)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::i8 [%0], %1, %2, %3, p;\n\t}"
                 :: "r"(d), "l"(a), "l"(b), "r"(i), "r"(1) : "memory");
    o[0] = 1;
}
'''


def _compile(arch: str):
    with tempfile.TemporaryDirectory() as td:
        src = os.path.join(td, "i8.cu")
        open(src, "w").write(SRC)
        return subprocess.run([NVCC, "-gencode", f"arch=compute_{arch},code=sm_{arch}", "-c", src,
                               "-o", os.path.join(td, "i8.o")], capture_output=True, text=True)


@pytest.mark.skipif(not os.path.exists(NVCC), reason="nvcc not installed")
def test_int8_tcgen05_mma_not_available_on_sm103a():
    r = _compile("103a")
    assert r.returncode != 0
    assert "kind::i8" in (r.stdout + r.stderr)
    assert _compile("100a").returncode == 0
