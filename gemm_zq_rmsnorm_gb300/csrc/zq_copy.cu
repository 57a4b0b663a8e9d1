// zq_copy.cu -- a copy by the SMs between any two buffers the device can
// address: device memory, or pinned host memory mapped into the device's
// address space (on a Grace-coupled GPU the SMs reach it coherently over the
// chip-to-chip link).  Meant for the small per-step activation copies of a
// decode step: a copy engine's start-up costs several microseconds there,
// which a kernel with one short round trip per thread does not pay.
#include "zq_async.cuh"
#include "zq_internal.cuh"

namespace zq {
namespace {

// 16-byte pieces, grid-stride; the bytes past the last whole piece by the
// first threads.  Both pointers 16-byte aligned.
__global__ void __launch_bounds__(256) copy16_kernel(uint4 *__restrict__ d, const uint4 *__restrict__ s,
                                                     size_t n16, uint8_t *__restrict__ dt,
                                                     const uint8_t *__restrict__ st, int tail)
{
    pdl_wait();   // the source may be the previous kernel's output
    pdl_launch_dependents();
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += stride) d[i] = s[i];
    const int t = (int)(blockIdx.x * blockDim.x + threadIdx.x);
    if (t < tail) dt[t] = st[t];
}

// Any alignment: byte by byte.
__global__ void __launch_bounds__(256) copy1_kernel(uint8_t *__restrict__ d, const uint8_t *__restrict__ s,
                                                    size_t n)
{
    pdl_wait();
    pdl_launch_dependents();
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) d[i] = s[i];
}

}  // namespace

// Up to one 256-thread block per 4 KB (16 bytes per thread), at most `sms`
// blocks: one round trip per thread for the activation sizes of a decode step.
cudaError_t launch_copy(void *dst, const void *src, size_t bytes, int sms, cudaStream_t st)
{
    if (bytes == 0) return cudaSuccess;
    const bool a16 = ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src)) & 15u) == 0;
    const size_t per_block = a16 ? 4096 : 256;
    size_t blocks = (bytes + per_block - 1) / per_block;
    if (blocks > (size_t)sms) blocks = (size_t)sms;
    if (a16) {
        const size_t n16 = bytes / 16;
        const int tail = (int)(bytes % 16);
        uint8_t *dt = static_cast<uint8_t *>(dst) + 16 * n16;
        const uint8_t *stail = static_cast<const uint8_t *>(src) + 16 * n16;
        return launch_pdl(copy16_kernel, dim3((unsigned)blocks), dim3(256), 0, st, static_cast<uint4 *>(dst),
                          static_cast<const uint4 *>(src), n16, dt, stail, tail);
    }
    return launch_pdl(copy1_kernel, dim3((unsigned)blocks), dim3(256), 0, st, static_cast<uint8_t *>(dst),
                      static_cast<const uint8_t *>(src), bytes);
}

}  // namespace zq
