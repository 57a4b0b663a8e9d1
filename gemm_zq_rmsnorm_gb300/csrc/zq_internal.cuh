// zq_internal.cuh -- helpers shared by the library's CUDA translation units.
// Internal to libzq.so; nothing here is exported.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "zq.h"

namespace zq {

constexpr int kQ4KBlockBytes = 144;   // one 256-weight super-block
constexpr int kQ4KBlockWeights = 256;

// Host-side launch descriptions (defined in the kernel TUs, called by the API).
cudaError_t launch_rmsnorm_q8_1(const float *x, const float *gamma, int B, int K,
                                float eps, zq_q8_1 out, cudaStream_t st);
// RMSNorm + Q8_1 with the token's row staged in shared memory (codes to *out
// when non-null) that also writes the batched projection's activation split
// when hi is non-null: hi/lo parts, token scales, s8 operand (K <= 32768,
// x 16-byte aligned).
cudaError_t launch_rmsnorm_q8_1_split(const float *x, const float *gamma, int B, int K, float eps,
                                      const zq_q8_1 *out, __half *hi, __half *lo, float *tscale, __half *s8x,
                                      cudaStream_t st);
cudaError_t launch_gemv(const void *W, const void *W2, int N, int K, zq_q8_1 a,
                        int B, float *y, float *y2, int32_t *isums,
                        cudaStream_t st);
// allow_split = false keeps one K range per tile (no partial-sum buffer).
cudaError_t launch_gemm_tc(const void *W, int N, int K, zq_q8_1 a, int B, float *y,
                           void *ws, bool allow_split, cudaStream_t st);
size_t gemm_tc_workspace_bytes(int N, int K, int B, bool allow_split = true);
cudaError_t launch_isums_tc(const void *W, int N, int K, zq_q8_1 a, int B,
                            int32_t *isums, void *ws, cudaStream_t st);
bool gemv_stream_supported(int K);
size_t noalloc_scratch_bytes();
cudaError_t launch_q4k_dequant_f16(const void *W, int N, int K, void *out, cudaStream_t st);
cudaError_t launch_q8_1_dequant_f16(zq_q8_1 a, int B, int K, void *out, cudaStream_t st);
// dense binary16 GEMM y[B][N] = X16[B][K] * W16[N][K]^T (f16_gemm_2sm.cu);
// part: split-K partial sums of f16_gemm_workspace_bytes
size_t f16_gemm_workspace_bytes(int N, int K, int B);
cudaError_t launch_f16_gemm(const void *W16, int N, int K, const void *X16, int B, float *y, float *part,
                            cudaStream_t st);
cudaError_t launch_gemm_noalloc(const void *W, int N, int K, zq_q8_1 a, int B, float *y, cudaStream_t st);
// Decode mat-vec job: up to kGemvMaxMats Q4_K matrices (N[m] x K) that read
// the same input vector.
constexpr int kGemvMaxMats = 4;
struct GemvJob {
    int nmat;
    const void *W[kGemvMaxMats];
    int N[kGemvMaxMats];
    float *y[kGemvMaxMats];
};
// input: Q8_1 codes of one token
cudaError_t launch_gemv_stream(const GemvJob &job, int K, zq_q8_1 a, cudaStream_t st);
// input: x and gamma, RMSNorm + Q8_1 computed in the kernel; or (silu) gate
// and up, Q8_1 of silu(gate) * up.  q8out, when non-null, receives the codes;
// pf/pf_bytes: optional range pulled into L2 for the next launch.
cudaError_t launch_gemv_stream_fused(const GemvJob &job, int K, const float *x, const float *gamma, float eps,
                                     bool silu, const zq_q8_1 *q8out, const void *pf, size_t pf_bytes,
                                     cudaStream_t st);
// Q5_K (176-byte blocks) and Q6_K (210-byte blocks) projections of B = 1 .. 16
// tokens of Q8_1 codes against one N x K matrix (K <= 32768); and the Q6_K
// mat-vec of one token given as x and gamma (RMSNorm + Q8_1 in the launch).
cudaError_t launch_q4k_tokens(const void *W, int N, int K, zq_q8_1 a, int B, float *y, cudaStream_t st);
cudaError_t launch_q4k_wait_expiry(const void *W, int N, int K, zq_q8_1 a, float *y, int withhold,
                                   uint64_t wait_ns, int ctas, cudaStream_t st);
cudaError_t launch_q5k_tokens(const void *W, int N, int K, zq_q8_1 a, int B, float *y, cudaStream_t st);
cudaError_t launch_q6k_tokens(const void *W, int N, int K, zq_q8_1 a, int B, float *y, cudaStream_t st);
cudaError_t launch_q6k_fused(const GemvJob &job, int K, const float *x, const float *gamma, float eps,
                             const zq_q8_1 *q8out, cudaStream_t st);
// Launch plan of the streamed mat-vec for a weight format (4, 5, 6 = Q4_K,
// Q5_K, Q6_K) and tokens per launch (1 or 4): false when it does not fit.
bool stream_plan_query(int fmt, int nt, int K, long long total_rows, int sms, int32_t *out);
cudaError_t launch_silu_mul_q8_1(const float *g, const float *u, int B, int K, zq_q8_1 out, cudaStream_t st);
// Throughput probes (kind 0: dp4a, 1: mma.sync m16n8k32 s8, 2: tcgen05 kind::f16
// 128 x 256 x 16); sink: device ints, one per thread (256 per block, 128 for kind 2).
cudaError_t launch_peak_probe(int kind, int blocks, int iters, int *sink, cudaStream_t st);
// Copy by the SMs (zq_copy): dst and src are device addresses.
cudaError_t launch_copy(void *dst, const void *src, size_t bytes, int sms, cudaStream_t st);

// Launch with programmatic dependent launch: the kernel may start while the
// previous kernel on the stream is still running.  Every kernel launched this
// way executes griddepcontrol.wait before it reads anything an earlier kernel
// may write and before it writes anything; only reads of data no kernel of
// the library writes (weights) and on-chip set-up may come first.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// Device-side error word of the current device (bit 0: a bounded wait in a
// pipelined kernel expired).  Valid after the first successful device check.
unsigned int *device_status_word();

int num_sms();

// ------------------------------------------------------------------ device
__device__ __forceinline__ uint4 ld_stream_u4(const void *p)
{
    // weights are read exactly once: do not keep them in L1
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint4 ld_cached_u4(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float h2f(uint16_t h)
{
    return __half2float(__ushort_as_half(h));
}

// Six-bit scale and min of sub-block j from the 12 packed scale bytes, given
// as three little-endian words s0 = S[0..3], s1 = S[4..7], s2 = S[8..11].
__device__ __forceinline__ void q4k_scale_min(uint32_t s0, uint32_t s1, uint32_t s2,
                                              int j, uint32_t &sc, uint32_t &m)
{
    if (j < 4) {
        sc = (s0 >> (8 * j)) & 63u;
        m = (s1 >> (8 * j)) & 63u;
    } else {
        const int k = 8 * (j - 4);
        const uint32_t b2 = (s2 >> k) & 0xFFu;
        sc = (b2 & 15u) | (((s0 >> k) >> 6 & 3u) << 4);
        m = (b2 >> 4) | (((s1 >> k) >> 6 & 3u) << 4);
    }
}

}  // namespace zq
