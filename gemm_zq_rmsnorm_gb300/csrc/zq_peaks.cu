// zq_peaks.cu -- throughput probes for the arithmetic the projection kernels
// can use on this GPU, timed by the caller: the packed int8 dot product
// (dp4a, the decode mat-vec's inner product), the legacy warp-level int8
// tensor-core MMA (mma.sync m16n8k32 s8), and the 5th-generation tensor-core
// MMA with binary16 operands (tcgen05 kind::f16, the batched projection's
// instruction).  The int8 tcgen05 MMA (kind::i8) is not available on sm_103a,
// so these rates are the denominators behind the prefill metric.  Each probe
// keeps its results live by writing one value per thread or CTA to `sink`.
#include <cuda.h>

#include "zq_cluster.cuh"
#include "zq_internal.cuh"
#include "zq_tc.cuh"

namespace zq {
namespace {

// 8 independent dp4a chains per thread, `iters` steps each.
__global__ void __launch_bounds__(256) probe_dp4a_kernel(int iters, int seed, int *sink)
{
    int acc[8];
    int a = seed + threadIdx.x, b = 0x01020304 ^ blockIdx.x;
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = j;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = __dp4a(a + j, b, acc[j]);
    }
    int s = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) s += acc[j];
    sink[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

// 4 independent m16n8k32 s8 MMAs per warp and step.
__global__ void __launch_bounds__(256) probe_mma_s8_kernel(int iters, int seed, int *sink)
{
    uint32_t a0 = seed + threadIdx.x, a1 = a0 * 3u, a2 = a0 * 5u, a3 = a0 * 7u, b0 = 0x01010101u, b1 = 0x02020202u;
    int c[4][4];
#pragma unroll
    for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int j = 0; j < 4; ++j) c[m][j] = 0;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int m = 0; m < 4; ++m)
            asm volatile(
                "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                "{%0,%1,%2,%3};"
                : "+r"(c[m][0]), "+r"(c[m][1]), "+r"(c[m][2]), "+r"(c[m][3])
                : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
    int s = 0;
#pragma unroll
    for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int j = 0; j < 4; ++j) s += c[m][j];
    sink[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

// One CTA per SM: one thread issues `iters` back-to-back 128 x 256 x 16
// binary16 MMAs (fp32 accumulate in tensor memory) on operands in shared
// memory, then waits for them (bounded) and reads one accumulator value.
constexpr int kProbeSmem = 2 * 128 * 128 + 2 * 256 * 128 + 1024;

// MMA shapes of the probe kinds 2.. (M = 128, K = 16): N, whether A is read
// from tensor memory (columns 128.., written once) instead of shared memory,
// and whether two warps issue at once (each `iters` MMAs into its own
// accumulator: columns 0.. and 64..)
__host__ __device__ constexpr int probe_tc_n(int kind) { return kind == 2 ? 256 : kind == 4 ? 16 : 32; }
__host__ __device__ constexpr bool probe_tc_ta(int kind) { return kind == 5; }
__host__ __device__ constexpr bool probe_tc_two(int kind) { return kind == 6; }
// kinds 8 (one CTA) and 9 (a pair): the issuing loop runs on all lanes of a
// warp and one elected lane issues each MMA
__host__ __device__ constexpr bool probe_tc_warp(int kind) { return kind == 8 || kind == 9; }


__global__ void __launch_bounds__(128, 1) probe_tc_f16_kernel(int kind, int iters, int *sink, unsigned int *status)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    __shared__ uint64_t bar;
    __shared__ uint32_t slot;
    const int warp = threadIdx.x >> 5;
    // operands: 128 rows (A) and 256 rows (B) of 64 binary16, small values
    for (int i = threadIdx.x; i < (2 * 128 * 128 + 2 * 256 * 128) / 4; i += blockDim.x)
        reinterpret_cast<uint32_t *>(sm)[i] = 0x3C003C00u;   // 1.0, 1.0
    fence_async_smem();
    if (threadIdx.x == 0) {
        mbar_init(&bar, probe_tc_two(kind) ? 2 : 1);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(&slot, 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = slot;
    if (probe_tc_ta(kind)) {
        // A in tensor memory: 128 lanes x 32 columns of binary16 pairs 1.0
        uint32_t one[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) one[i] = 0x3C003C00u;
        tmem_st16(tmem + ((uint32_t)(32 * warp) << 16) + 128u, one);
        tmem_st16(tmem + ((uint32_t)(32 * warp) << 16) + 144u, one);
        tmem_wait_st();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (probe_tc_warp(kind)) {
        if (warp == 0) {
            const uint32_t base = smem_u32(sm);
            const uint64_t ad = smem_desc(base, 16, 1024, kLayoutSw128);
            const uint64_t bd = smem_desc(base + 2 * 128 * 128, 16, 1024, kLayoutSw128);
            const uint32_t idesc = idesc_f16_f32(128, 32);
            for (int it = 0; it < iters; ++it) {
                if (elect_one()) mma_f16(tmem, ad + 2 * (it & 3), bd + 2 * (it & 3), idesc, it > 0 ? 1u : 0u);
                __syncwarp();
            }
            if (elect_one()) mma_commit(&bar);
            __syncwarp();
            if ((threadIdx.x & 31) == 0) mbar_wait(&bar, 0, status);
            __syncwarp();
        }
    } else if (threadIdx.x == 0 || (probe_tc_two(kind) && threadIdx.x == 32)) {
        const uint32_t d = tmem + (threadIdx.x ? 64u : 0u);
        const uint32_t base = smem_u32(sm);
        const uint64_t ad = smem_desc(base, 16, 1024, kLayoutSw128);
        const uint64_t bd = smem_desc(base + 2 * 128 * 128, 16, 1024, kLayoutSw128);
        const uint32_t idesc = idesc_f16_f32(128, (uint32_t)probe_tc_n(kind));
        if (probe_tc_ta(kind)) {
            for (int it = 0; it < iters; ++it)
                mma_f16_ta(d, tmem + 128u + 8u * (it & 3), bd + 2 * (it & 3), idesc, it > 0 ? 1u : 0u);
        } else {
            for (int it = 0; it < iters; ++it)
                mma_f16(d, ad + 2 * (it & 3), bd + 2 * (it & 3), idesc, it > 0 ? 1u : 0u);
        }
        mma_commit(&bar);
        mbar_wait(&bar, 0, status);
    }
    __syncthreads();
    tc_fence_after();
    uint32_t r[16];
    tmem_ld16(tmem + ((uint32_t)(32 * warp) << 16), r);
    tmem_wait_ld();
    sink[blockIdx.x * blockDim.x + threadIdx.x] = (int)r[0];
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

// Kind 7: a CTA pair; one thread of the even CTA issues `iters` 256 x 32 x 16
// MMAs (cta_group::2: 128 rows in each SM's tensor memory), operands in each
// CTA's shared memory.
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(128, 1)
probe_tc_pair_kernel(int iters, int warpwide, int a_tmem, int *sink, unsigned int *status)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    __shared__ uint64_t bar;
    __shared__ uint32_t slot;
    const int warp = threadIdx.x >> 5;
    const uint32_t rank = cluster_rank();
    for (int i = threadIdx.x; i < (2 * 128 * 128 + 2 * 256 * 128) / 4; i += blockDim.x)
        reinterpret_cast<uint32_t *>(sm)[i] = 0x3C003C00u;
    fence_async_smem();
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc_pair(&slot, 256);
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem = slot;
    if (a_tmem) {
        // A in tensor memory: 128 lanes x 32 columns of binary16 pairs 1.0
        uint32_t one[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) one[i] = 0x3C003C00u;
        tmem_st16(tmem + ((uint32_t)(32 * warp) << 16) + 128u, one);
        tmem_st16(tmem + ((uint32_t)(32 * warp) << 16) + 144u, one);
        tmem_wait_st();
    }
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    if (rank == 0 && warpwide && warp == 0) {
        const uint32_t base = smem_u32(sm);
        const uint64_t ad = smem_desc(base, 16, 1024, kLayoutSw128);
        const uint64_t bd = smem_desc(base + 2 * 128 * 128, 16, 1024, kLayoutSw128);
        const uint32_t idesc = idesc_f16_f32(256, 32);
        for (int it = 0; it < iters; ++it) {
            if (elect_one()) {
                if (a_tmem)
                    mma_f16_pair_ta(tmem, tmem + 128u + 8u * (it & 3), bd + 2 * (it & 3), idesc, it > 0 ? 1u : 0u);
                else
                    mma_f16_pair(tmem, ad + 2 * (it & 3), bd + 2 * (it & 3), idesc, it > 0 ? 1u : 0u);
            }
            __syncwarp();
        }
        if (elect_one()) mma_commit_pair_mc(&bar, 3);
        __syncwarp();
    } else if (rank == 0 && !warpwide && threadIdx.x == 0) {
        const uint32_t base = smem_u32(sm);
        const uint64_t ad = smem_desc(base, 16, 1024, kLayoutSw128);
        const uint64_t bd = smem_desc(base + 2 * 128 * 128, 16, 1024, kLayoutSw128);
        const uint32_t idesc = idesc_f16_f32(256, 32);
        for (int it = 0; it < iters; ++it)
            mma_f16_pair(tmem, ad + 2 * (it & 3), bd + 2 * (it & 3), idesc, it > 0 ? 1u : 0u);
        mma_commit_pair_mc(&bar, 3);
    }
    if (threadIdx.x == 0) {
        // both CTAs wait for the commit that reaches them (bounded)
        const uint64_t t0 = global_ns();
        while (!mbar_try_wait_cl_sleep(&bar, 0, kSleepNs)) {
            if (global_ns() - t0 >= kWaitLimitNs) {
                flag_timeout(status);
                break;
            }
        }
    }
    __syncthreads();
    tc_fence_after();
    uint32_t r[16];
    tmem_ld16(tmem + ((uint32_t)(32 * warp) << 16), r);
    tmem_wait_ld();
    sink[blockIdx.x * blockDim.x + threadIdx.x] = (int)r[0];
    tc_fence_before();
    cluster_sync();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, 256);
    }
}

size_t g_attr_bytes[64];
size_t g_attr_pair[64];

}  // namespace

cudaError_t launch_peak_probe(int kind, int blocks, int iters, int *sink, cudaStream_t st)
{
    if (kind == 0) {
        probe_dp4a_kernel<<<blocks, 256, 0, st>>>(iters, 1, sink);
    } else if (kind == 1) {
        probe_mma_s8_kernel<<<blocks, 256, 0, st>>>(iters, 1, sink);
    } else {
        int dev = 0;
        cudaGetDevice(&dev);
        if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
        if (g_attr_bytes[dev] < (size_t)kProbeSmem) {
            cudaError_t e =
                cudaFuncSetAttribute(probe_tc_f16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kProbeSmem);
            if (e != cudaSuccess) return e;
            g_attr_bytes[dev] = kProbeSmem;
        }
        if (kind == 7 || kind == 9 || kind == 10) {
            if (g_attr_pair[dev] < (size_t)kProbeSmem) {
                cudaError_t e = cudaFuncSetAttribute(probe_tc_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                     kProbeSmem);
                if (e != cudaSuccess) return e;
                g_attr_pair[dev] = kProbeSmem;
            }
            probe_tc_pair_kernel<<<2 * (blocks / 2), 128, kProbeSmem, st>>>(iters, kind >= 9 ? 1 : 0, kind == 10 ? 1 : 0,
                                                                             sink, device_status_word());
        } else {
            probe_tc_f16_kernel<<<blocks, 128, kProbeSmem, st>>>(kind, iters, sink, device_status_word());
        }
    }
    return cudaGetLastError();
}

}  // namespace zq
