"""Python binding of libzq.so, the GB300 quantized-projection library.

Argument marshalling only: every step of the path (RMSNorm + Q8_1 packing,
Q4_K x Q8_1 mat-vec / paired mat-vec / batched GEMM) runs in the library's
CUDA kernels.  PyTorch supplies device memory and the current stream.  There
is no CPU fallback: if libzq.so is missing or the device is not sm_103, every
call raises.

The entry points mirror the C ABI of include/zq.h one to one.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libzq.so")

ZQ_OK = 0
DEVICE_WAIT_EXPIRED = 1   # bit of the device status word: a bounded wait expired
STATUS_NAMES = {0: "ZQ_OK", -1: "ZQ_ERR_ARG", -2: "ZQ_ERR_SHAPE", -3: "ZQ_ERR_ALIGN",
                -4: "ZQ_ERR_CUDA", -5: "ZQ_ERR_DEVICE", -6: "ZQ_ERR_WORKSPACE"}

EXPORTS = ("zq_rmsnorm_q8_1", "zq_q4k_gemv", "zq_q4k_gemv_pair", "zq_q4k_gemm",
           "zq_q4k_gemm_workspace_bytes", "zq_q4k_bytes", "zq_q8_1_bytes",
           "zq_status_string", "zq_last_error", "zq_version", "zq_debug_q4k_isums",
           "zq_device_status", "zq_q4k_gemm_noalloc", "zq_q4k_gemv_multi", "zq_rmsnorm_q4k_gemv",
           "zq_q4k_dequant_f16", "zq_silu_mul_q8_1", "zq_silu_q4k_gemv",
           "zq_q5k_gemm", "zq_q6k_gemm", "zq_q5k_gemv", "zq_q6k_gemv", "zq_rmsnorm_q6k_gemv",
           "zq_q5k_bytes", "zq_q6k_bytes", "zq_debug_stream_plan", "zq_debug_peak_probe",
           "zq_debug_wait_expiry", "zq_q8_1_dequant_f16", "zq_f16_gemm_workspace_bytes", "zq_f16_gemm",
           "zq_rmsnorm_q4k_gemm", "zq_copy")


class ZQError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class _Q8(ctypes.Structure):
    _fields_ = [("qs", ctypes.c_void_p), ("d", ctypes.c_void_p), ("s", ctypes.c_void_p)]


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libzq.so (built by gemm_zq_rmsnorm_gb300/build.py); raise if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libzq.so not found at {path}: build it with "
                           "`python gemm_zq_rmsnorm_gb300/build.py` (needs nvcc)")
    lib = ctypes.CDLL(path)
    P, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    sig = {
        "zq_rmsnorm_q8_1": ([P, P, i, i, f, _Q8, P], i),
        "zq_q4k_gemv": ([P, i, i, _Q8, P, P], i),
        "zq_q4k_gemv_pair": ([P, P, i, i, _Q8, P, P, P], i),
        "zq_q4k_gemm": ([P, i, i, _Q8, i, P, P, sz, P], i),
        "zq_q4k_gemm_workspace_bytes": ([i, i, i], sz),
        "zq_q4k_bytes": ([i, i], sz),
        "zq_q8_1_bytes": ([i, i], sz),
        "zq_status_string": ([i], ctypes.c_char_p),
        "zq_last_error": ([], ctypes.c_char_p),
        "zq_version": ([], i),
        "zq_debug_q4k_isums": ([P, i, i, _Q8, i, P, i, P, sz, P], i),
        "zq_device_status": ([P, i], i),
        "zq_q4k_gemm_noalloc": ([P, i, i, _Q8, i, P, P], i),
        "zq_q4k_gemv_multi": ([i, P, P, i, _Q8, P, P], i),
        "zq_q4k_dequant_f16": ([P, i, i, P, P], i),
        "zq_silu_mul_q8_1": ([P, P, i, i, _Q8, P], i),
        "zq_silu_q4k_gemv": ([P, P, i, i, P, P, P, ctypes.POINTER(_Q8), P, sz, P], i),
        "zq_rmsnorm_q4k_gemv": ([P, P, f, i, i, P, P, P, ctypes.POINTER(_Q8), P, sz, P], i),
        "zq_q5k_gemm": ([P, i, i, _Q8, i, P, P], i),
        "zq_q6k_gemm": ([P, i, i, _Q8, i, P, P], i),
        "zq_copy": ([P, P, sz, P], i),
        "zq_q5k_gemv": ([P, i, i, _Q8, P, P], i),
        "zq_q6k_gemv": ([P, i, i, _Q8, P, P], i),
        "zq_rmsnorm_q6k_gemv": ([P, P, f, i, P, i, P, ctypes.POINTER(_Q8), P], i),
        "zq_q5k_bytes": ([i, i], sz),
        "zq_q6k_bytes": ([i, i], sz),
        "zq_debug_stream_plan": ([i, i, i, ctypes.c_longlong, i, P], i),
        "zq_debug_peak_probe": ([i, i, i, P, P], i),
        "zq_debug_wait_expiry": ([P, i, i, _Q8, P, i, ctypes.c_uint, i, P], i),
        "zq_q8_1_dequant_f16": ([_Q8, i, i, P, P], i),
        "zq_f16_gemm_workspace_bytes": ([i, i, i], sz),
        "zq_f16_gemm": ([P, i, i, P, i, P, P, sz, P], i),
        "zq_rmsnorm_q4k_gemm": ([P, P, f, i, i, P, i, P, ctypes.POINTER(_Q8), P, sz, P], i),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def _check(status: int):
    if status != ZQ_OK:
        raise ZQError(status, load().zq_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


@dataclasses.dataclass
class Q8_1:
    """Planar Q8_1 activations: qs int8 [B][K], d/s binary16 [B][K/32]."""
    qs: torch.Tensor
    d: torch.Tensor
    s: torch.Tensor

    @property
    def B(self) -> int:
        return self.qs.shape[0]

    @property
    def K(self) -> int:
        return self.qs.shape[1]

    def _c(self) -> _Q8:
        return _Q8(self.qs.data_ptr(), self.d.data_ptr(), self.s.data_ptr())

    def rows(self, t0: int, t1: int) -> "Q8_1":
        return Q8_1(self.qs[t0:t1], self.d[t0:t1], self.s[t0:t1])


def empty_q8_1(B: int, K: int, device="cuda") -> Q8_1:
    return Q8_1(torch.empty((B, K), dtype=torch.int8, device=device),
                torch.empty((B, K // 32), dtype=torch.float16, device=device),
                torch.empty((B, K // 32), dtype=torch.float16, device=device))


def q4k_bytes(N: int, K: int) -> int:
    return int(load().zq_q4k_bytes(N, K))


def gemm_workspace_bytes(N: int, K: int, B: int) -> int:
    return int(load().zq_q4k_gemm_workspace_bytes(N, K, B))


def rmsnorm_q8_1(x: torch.Tensor, gamma: torch.Tensor, eps: float, out: Q8_1 | None = None,
                 stream=None) -> Q8_1:
    """Fused RMSNorm + Q8_1 pack of x fp32 [B][K] (see zq_rmsnorm_q8_1)."""
    lib = load()
    B, K = x.shape
    if out is None:
        out = empty_q8_1(B, K, x.device)
    _check(lib.zq_rmsnorm_q8_1(_ptr(x), _ptr(gamma), B, K, float(eps), out._c(), _stream(stream)))
    return out


def _job_arrays(Ws, Ns, ys):
    n = len(Ws)
    if not (len(Ns) == n and len(ys) == n):
        raise ValueError("W, N and y lists must have the same length")
    W_arr = (ctypes.c_void_p * max(n, 1))(*[w.data_ptr() for w in Ws])
    N_arr = (ctypes.c_int * max(n, 1))(*[int(v) for v in Ns])
    y_arr = (ctypes.c_void_p * max(n, 1))(*[y.data_ptr() for y in ys])
    return n, W_arr, N_arr, y_arr


def q4k_gemv_multi(Ws, Ns, K: int, a: Q8_1, ys=None, stream=None):
    """y[m] = W[m] a for up to four matrices sharing one Q8_1 input (see
    zq_q4k_gemv_multi); returns the list of outputs."""
    lib = load()
    if ys is None:
        ys = [torch.empty(int(n), dtype=torch.float32, device=a.qs.device) for n in Ns]
    n, W_arr, N_arr, y_arr = _job_arrays(Ws, Ns, ys)
    _check(lib.zq_q4k_gemv_multi(n, ctypes.cast(W_arr, ctypes.c_void_p), ctypes.cast(N_arr, ctypes.c_void_p), K,
                                 a._c(), ctypes.cast(y_arr, ctypes.c_void_p), _stream(stream)))
    return ys


def rmsnorm_q4k_gemv(x: torch.Tensor, gamma: torch.Tensor, eps: float, Ws, Ns, ys=None,
                     q8_out: Q8_1 | None = None, stream=None, l2_prefetch: torch.Tensor | None = None,
                     l2_prefetch_bytes: int = 0):
    """RMSNorm + Q8_1 of one token x fp32 [K] (or [1][K]) fused with the
    mat-vecs of up to four matrices (see zq_rmsnorm_q4k_gemv); l2_prefetch
    optionally names the bytes the next launch will read."""
    lib = load()
    K = x.shape[-1]
    if ys is None:
        ys = [torch.empty(int(n), dtype=torch.float32, device=x.device) for n in Ns]
    n, W_arr, N_arr, y_arr = _job_arrays(Ws, Ns, ys)
    q8 = ctypes.byref(q8_out._c()) if q8_out is not None else None
    _check(lib.zq_rmsnorm_q4k_gemv(_ptr(x), _ptr(gamma), float(eps), K, n, ctypes.cast(W_arr, ctypes.c_void_p),
                                   ctypes.cast(N_arr, ctypes.c_void_p), ctypes.cast(y_arr, ctypes.c_void_p), q8,
                                   _ptr(l2_prefetch),
                                   int(l2_prefetch_bytes if l2_prefetch is not None else 0), _stream(stream)))
    return ys


def q4k_dequant_f16(W: torch.Tensor, N: int, K: int, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Q4_K N x K -> binary16 [N][K] (see zq_q4k_dequant_f16)."""
    lib = load()
    if out is None:
        out = torch.empty((N, K), dtype=torch.float16, device=W.device)
    _check(lib.zq_q4k_dequant_f16(_ptr(W), N, K, _ptr(out), _stream(stream)))
    return out


def q8_1_dequant_f16(a: Q8_1, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Q8_1 planes of B tokens -> binary16 [B][K], x = q8 * d8 (see zq_q8_1_dequant_f16)."""
    lib = load()
    B, K = a.B, a.K
    if out is None:
        out = torch.empty((B, K), dtype=torch.float16, device=a.qs.device)
    _check(lib.zq_q8_1_dequant_f16(a._c(), B, K, _ptr(out), _stream(stream)))
    return out


def f16_gemm_workspace_bytes(N: int, K: int, B: int) -> int:
    return int(load().zq_f16_gemm_workspace_bytes(N, K, B))


def f16_gemm(W16: torch.Tensor, N: int, K: int, X16: torch.Tensor, B: int, y: torch.Tensor | None = None,
             workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y[B][N] = X16 @ W16^T on the tensor cores (see zq_f16_gemm)."""
    lib = load()
    dev = W16.device
    if y is None:
        y = torch.empty((B, N), dtype=torch.float32, device=dev)
    need = f16_gemm_workspace_bytes(N, K, B)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.zq_f16_gemm(_ptr(W16), N, K, _ptr(X16), B, _ptr(y), _ptr(workspace), wbytes, _stream(stream)))
    return y


def silu_mul_q8_1(gate: torch.Tensor, up: torch.Tensor, out: Q8_1 | None = None, stream=None) -> Q8_1:
    """Q8_1 of silu(gate) * up, fp32 [B][K] each (see zq_silu_mul_q8_1)."""
    lib = load()
    B, K = gate.shape
    if out is None:
        out = empty_q8_1(B, K, gate.device)
    _check(lib.zq_silu_mul_q8_1(_ptr(gate), _ptr(up), B, K, out._c(), _stream(stream)))
    return out


def silu_q4k_gemv(gate: torch.Tensor, up: torch.Tensor, Ws, Ns, ys=None, q8_out: Q8_1 | None = None,
                  stream=None, l2_prefetch: torch.Tensor | None = None, l2_prefetch_bytes: int = 0):
    """Q8_1 of silu(gate) * up for one token (fp32 [K] each) fused with the
    mat-vecs of up to four matrices (see zq_silu_q4k_gemv)."""
    lib = load()
    K = gate.shape[-1]
    if ys is None:
        ys = [torch.empty(int(n), dtype=torch.float32, device=gate.device) for n in Ns]
    n, W_arr, N_arr, y_arr = _job_arrays(Ws, Ns, ys)
    q8 = ctypes.byref(q8_out._c()) if q8_out is not None else None
    _check(lib.zq_silu_q4k_gemv(_ptr(gate), _ptr(up), K, n, ctypes.cast(W_arr, ctypes.c_void_p),
                                ctypes.cast(N_arr, ctypes.c_void_p), ctypes.cast(y_arr, ctypes.c_void_p), q8,
                                _ptr(l2_prefetch), int(l2_prefetch_bytes if l2_prefetch is not None else 0),
                                _stream(stream)))
    return ys


def q4k_gemv(W: torch.Tensor, N: int, K: int, a: Q8_1, y: torch.Tensor | None = None,
             stream=None) -> torch.Tensor:
    lib = load()
    if y is None:
        y = torch.empty(N, dtype=torch.float32, device=a.qs.device)
    _check(lib.zq_q4k_gemv(_ptr(W), N, K, a._c(), _ptr(y), _stream(stream)))
    return y


def q4k_gemv_pair(Wg: torch.Tensor, Wu: torch.Tensor, N: int, K: int, a: Q8_1,
                  y_gate: torch.Tensor | None = None, y_up: torch.Tensor | None = None,
                  stream=None):
    lib = load()
    dev = a.qs.device
    if y_gate is None:
        y_gate = torch.empty(N, dtype=torch.float32, device=dev)
    if y_up is None:
        y_up = torch.empty(N, dtype=torch.float32, device=dev)
    _check(lib.zq_q4k_gemv_pair(_ptr(Wg), _ptr(Wu), N, K, a._c(), _ptr(y_gate), _ptr(y_up),
                                _stream(stream)))
    return y_gate, y_up


def q4k_gemm(W: torch.Tensor, N: int, K: int, a: Q8_1, B: int | None = None,
             y: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
             stream=None) -> torch.Tensor:
    lib = load()
    B = a.B if B is None else B
    dev = a.qs.device
    if y is None:
        y = torch.empty((B, N), dtype=torch.float32, device=dev)
    need = gemm_workspace_bytes(N, K, B)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.zq_q4k_gemm(_ptr(W), N, K, a._c(), B, _ptr(y), _ptr(workspace), wbytes,
                           _stream(stream)))
    return y


def rmsnorm_q4k_gemm(x: torch.Tensor, gamma: torch.Tensor, eps: float, W: torch.Tensor, N: int,
                     y: torch.Tensor | None = None, q8_out: Q8_1 | None = None,
                     workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """RMSNorm + Q8_1 of x [B][K] and the projection y [B][N] in one call (see zq_rmsnorm_q4k_gemm)."""
    lib = load()
    B, K = x.shape
    dev = x.device
    if y is None:
        y = torch.empty((B, N), dtype=torch.float32, device=dev)
    if q8_out is None and 2 <= B <= 4:
        q8_out = empty_q8_1(B, K, dev)
    need = gemm_workspace_bytes(N, K, B)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    q8 = ctypes.byref(q8_out._c()) if q8_out is not None else None
    _check(lib.zq_rmsnorm_q4k_gemm(_ptr(x), _ptr(gamma), float(eps), B, K, _ptr(W), N, _ptr(y), q8,
                                   _ptr(workspace), wbytes, _stream(stream)))
    return y


def q4k_gemm_noalloc(W: torch.Tensor, N: int, K: int, a: Q8_1, B: int | None = None,
                     y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """zq_q4k_gemm with the library's built-in scratch (no workspace; see zq.h)."""
    lib = load()
    B = a.B if B is None else B
    if y is None:
        y = torch.empty((B, N), dtype=torch.float32, device=a.qs.device)
    _check(lib.zq_q4k_gemm_noalloc(_ptr(W), N, K, a._c(), B, _ptr(y), _stream(stream)))
    return y


def kq_bytes(fmt: str, N: int, K: int) -> int:
    """Storage bytes of an N x K matrix of format "q4k", "q5k" or "q6k"."""
    fn = {"q4k": load().zq_q4k_bytes, "q5k": load().zq_q5k_bytes, "q6k": load().zq_q6k_bytes}[fmt]
    return int(fn(N, K))


def kq_gemm(fmt: str, W: torch.Tensor, N: int, K: int, a: Q8_1, B: int | None = None,
            y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y [B][N] for a Q5_K ("q5k") or Q6_K ("q6k") matrix and 1 <= B <= 16
    tokens (see zq_q5k_gemm / zq_q6k_gemm; B = 1 goes through *_gemv)."""
    lib = load()
    B = a.B if B is None else B
    if y is None:
        y = torch.empty((B, N), dtype=torch.float32, device=a.qs.device)
    if B == 1:
        fn = {"q5k": lib.zq_q5k_gemv, "q6k": lib.zq_q6k_gemv}[fmt]
        _check(fn(_ptr(W), N, K, a._c(), _ptr(y), _stream(stream)))
    else:
        fn = {"q5k": lib.zq_q5k_gemm, "q6k": lib.zq_q6k_gemm}[fmt]
        _check(fn(_ptr(W), N, K, a._c(), B, _ptr(y), _stream(stream)))
    return y


def rmsnorm_q6k_gemv(x: torch.Tensor, gamma: torch.Tensor, eps: float, W: torch.Tensor, N: int,
                     y: torch.Tensor | None = None, q8_out: Q8_1 | None = None, stream=None) -> torch.Tensor:
    """RMSNorm + Q8_1 of one token x fp32 [K] fused with a Q6_K mat-vec (the LM
    head after the final norm; see zq_rmsnorm_q6k_gemv)."""
    lib = load()
    K = x.shape[-1]
    if y is None:
        y = torch.empty(N, dtype=torch.float32, device=x.device)
    q8 = ctypes.byref(q8_out._c()) if q8_out is not None else None
    _check(lib.zq_rmsnorm_q6k_gemv(_ptr(x), _ptr(gamma), float(eps), K, _ptr(W), N, _ptr(y), q8, _stream(stream)))
    return y


def debug_stream_plan(wtype: int, ntok: int, K: int, total_rows: int, sms: int = 152) -> dict:
    """Launch plan of the streamed mat-vec (host-side; see zq_debug_stream_plan)."""
    out = (ctypes.c_int32 * 8)()
    _check(load().zq_debug_stream_plan(wtype, ntok, K, total_rows, sms, ctypes.cast(out, ctypes.c_void_p)))
    keys = ("R", "P", "CB", "nseg", "wl", "stage_alloc", "smem", "rowbytes")
    return dict(zip(keys, list(out)))


def copy(dst: torch.Tensor, src: torch.Tensor, stream=None) -> torch.Tensor:
    """Copy src into dst (same byte size, both contiguous) with the GPU's SMs
    (zq_copy): each may live on this GPU or in pinned host memory."""
    if not (dst.is_contiguous() and src.is_contiguous()):
        raise ValueError("copy: dst and src must be contiguous")
    nbytes = src.numel() * src.element_size()
    if dst.numel() * dst.element_size() != nbytes:
        raise ValueError("copy: dst and src differ in size")
    _check(load().zq_copy(_ptr(dst), _ptr(src), nbytes, _stream(stream)))
    return dst


def device_status(clear: bool = False) -> int:
    """Device-side error word (bit 0: a bounded wait in a pipelined kernel expired)."""
    flags = ctypes.c_uint(0)
    _check(load().zq_device_status(ctypes.byref(flags), int(clear)))
    return int(flags.value)


def debug_q4k_isums(W: torch.Tensor, N: int, K: int, a: Q8_1, path: int = 0,
                    workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Exact sub-block integer sums [B][N][K/32] from the kernels' own inner
    products (path 0: dp4a mat-vec; 1: prefill tensor cores; 2: chunk tensor cores)."""
    lib = load()
    B = a.B
    dev = a.qs.device
    isums = torch.empty((B, N, K // 32), dtype=torch.int32, device=dev)
    need = 2 * B * K if path else 0   # the binary16 copy of the codes (paths 1, 2)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.zq_debug_q4k_isums(_ptr(W), N, K, a._c(), B, _ptr(isums), path, _ptr(workspace),
                                  wbytes, _stream(stream)))
    return isums


def debug_wait_expiry(W: torch.Tensor, N: int, K: int, a: Q8_1, y: torch.Tensor, withhold_stage: int,
                      wait_us: int = 1000, ctas: int = 1, stream=None) -> None:
    """One streamed mat-vec launch whose producers withhold a stage and whose
    waits give up after wait_us (see zq_debug_wait_expiry); the expiry shows
    in device_status()."""
    _check(load().zq_debug_wait_expiry(_ptr(W), N, K, a._c(), _ptr(y), withhold_stage, wait_us, ctas,
                                       _stream(stream)))


# operations per probe launch, by kind (zq_debug_peak_probe)
PROBE_KINDS = {0: "dp4a", 1: "mma.sync m16n8k32 s8", 2: "tcgen05.mma kind::f16 128x256x16",
               3: "tcgen05.mma kind::f16 128x32x16", 4: "tcgen05.mma kind::f16 128x16x16",
               5: "tcgen05.mma kind::f16 128x32x16, A in tensor memory",
               6: "tcgen05.mma kind::f16 128x32x16, two issuing warps per SM",
               7: "tcgen05.mma kind::f16 256x32x16, CTA pair",
               8: "tcgen05.mma kind::f16 128x32x16, warp-wide loop, elected lane",
               9: "tcgen05.mma kind::f16 256x32x16, CTA pair, warp-wide loop, elected lane",
               10: "tcgen05.mma kind::f16 256x32x16, CTA pair, warp-wide loop, A in tensor memory"}


def probe_ops(kind: int, blocks: int, iters: int) -> int:
    if kind == 0:
        return blocks * 256 * iters * 8 * 8
    if kind == 1:
        return blocks * 8 * iters * 4 * 2 * 16 * 8 * 32
    if kind == 6:
        return blocks * 2 * iters * 2 * 128 * 32 * 16
    if kind in (7, 9, 10):
        return (blocks // 2) * iters * 2 * 256 * 32 * 16
    n = {2: 256, 4: 16}.get(kind, 32)
    return blocks * iters * 2 * 128 * n * 16


def debug_peak_probe(kind: int, blocks: int, iters: int, sink: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """One launch of a throughput probe (see zq.h); returns the sink."""
    if sink is None:
        sink = torch.empty(blocks * 256, dtype=torch.int32, device="cuda")
    _check(load().zq_debug_peak_probe(kind, blocks, iters, _ptr(sink), _stream(stream)))
    return sink
