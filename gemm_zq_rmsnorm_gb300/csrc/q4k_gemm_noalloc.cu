// q4k_gemm_noalloc.cu -- zq_q4k_gemm without a caller-supplied workspace.
//
// The batched projection needs scratch device memory (the binary16 hi/lo
// split of the activations that the tensor cores read, and a per-token
// scale).  zq_q4k_gemm takes it from the caller.  Some callers have no device
// memory to hand over: engines that own every byte of device memory in a
// fixed arena and forbid allocation after start-up, and plugins invoked by a
// host framework that gives them no allocator.  For them this file keeps a
// fixed scratch buffer in a file-scope device array, sized for the largest
// shape the library's workloads use (a 512-token prefill of a 17408-wide
// projection input), and never allocates anything.
#include <mutex>

#include "zq_internal.cuh"

namespace zq {
namespace {

// Bytes of the shared scratch: 4 * B * K (hi and lo halves), B * K / 8 (the
// scaled block sums of the 2-SM kernel) and 4 * B (the token scales), each
// padded to 256 bytes, for B * K <= 10 Mi.
constexpr size_t kNoAllocScratchBytes = (42u << 20) + (256u << 10);

// One array per device that loads the library; it lives until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDev = 64;
void *g_scratch_addr[kMaxDev];
std::mutex g_scratch_mu;

// The array's host-side name is only a stand-in for the device symbol; the
// address a kernel may use is looked up once per device, with that device
// current.
cudaError_t scratch_for_current_device(void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

size_t noalloc_scratch_bytes() { return kNoAllocScratchBytes; }

cudaError_t launch_gemm_noalloc(const void *W, int N, int K, zq_q8_1 a, int B, float *y, cudaStream_t st)
{
    void *ws = nullptr;
    cudaError_t e = scratch_for_current_device(&ws);
    if (e != cudaSuccess) return e;
    // one K range per tile: the fixed array holds no split-K partial sums
    return launch_gemm_tc(W, N, K, a, B, y, ws, false, st);
}

}  // namespace zq
