// rmsnorm_q8_1.cu -- fused RMSNorm + Q8_1 activation packing.
//
// ZINC docs "ROCm backend", "Build and verify": RMS normalisation and Q8
// activation packing share one wide per-token kernel, saving a second read of
// the activations and a launch.
//
// One CTA of 256 threads per token.  Thread t owns the 32-element blocks
// b = t, t+256, t+512, ... of its token, which is exactly the slot layout of
// the fixed summation order of the library's definition (per-block fused
// multiply-add chain, per-slot sum over b = t mod 256, pairwise tree over the
// 256 slots).  Every floating-point step is an explicitly rounded IEEE fp32
// operation (__fmaf_rn, __fadd_rn, __fmul_rn, __fdiv_rn, __fsqrt_rn), so the
// codes and scales are reproducible bit for bit on any conforming
// implementation of the same definition.
//
// HBM roofline: reads B*K*4 bytes of x (+ K*4 of gamma, cached), writes
// B*K*(1 + 4/32) bytes.  The kernel is tiny next to the projections that
// consume its output.
#include "zq_internal.cuh"

namespace zq {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
rmsnorm_q8_1_kernel(const float *__restrict__ x, const float *__restrict__ gamma,
                    int K, float eps, int8_t *__restrict__ qs,
                    __half *__restrict__ dq, __half *__restrict__ sq)
{
    __shared__ float slot_s[kThreads];
    __shared__ float r_s;

    const int t = threadIdx.x;
    const int nblk = K >> 5;
    const float *xt = x + (size_t)blockIdx.x * K;

    // pass 1: slot t = sum over its blocks of the per-block fma chain
    float slot = 0.0f;
    for (int b = t; b < nblk; b += kThreads) {
        const float4 *p = reinterpret_cast<const float4 *>(xt + 32 * b);
        float part = 0.0f;
#pragma unroll
        for (int v = 0; v < 8; ++v) {
            const float4 f = __ldg(p + v);
            part = __fmaf_rn(f.x, f.x, part);
            part = __fmaf_rn(f.y, f.y, part);
            part = __fmaf_rn(f.z, f.z, part);
            part = __fmaf_rn(f.w, f.w, part);
        }
        slot = __fadd_rn(slot, part);
    }
    slot_s[t] = slot;
    __syncthreads();
    // pairwise tree, off = 128 .. 32 through shared memory
#pragma unroll
    for (int off = 128; off >= 32; off >>= 1) {
        if (t < off) slot_s[t] = __fadd_rn(slot_s[t], slot_s[t + off]);
        __syncthreads();
    }
    if (t < 32) {
        float v = slot_s[t];
        // off = 16 .. 1 within the first warp: lane l < off adds lane l + off
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) v = __fadd_rn(v, __shfl_down_sync(0xffffffffu, v, off));
        if (t == 0) {
            const float mean = __fdiv_rn(v, (float)K);
            r_s = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, eps)));
        }
    }
    __syncthreads();
    const float r = r_s;

    // pass 2: normalise and pack each owned block
    for (int b = t; b < nblk; b += kThreads) {
        const float4 *p = reinterpret_cast<const float4 *>(xt + 32 * b);
        const float4 *g = reinterpret_cast<const float4 *>(gamma + 32 * b);
        float xh[32];
        float amax = 0.0f;
#pragma unroll
        for (int v = 0; v < 8; ++v) {
            const float4 f = __ldg(p + v);
            const float4 w = __ldg(g + v);
            xh[4 * v + 0] = __fmul_rn(__fmul_rn(f.x, r), w.x);
            xh[4 * v + 1] = __fmul_rn(__fmul_rn(f.y, r), w.y);
            xh[4 * v + 2] = __fmul_rn(__fmul_rn(f.z, r), w.z);
            xh[4 * v + 3] = __fmul_rn(__fmul_rn(f.w, r), w.w);
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(xh[i]));
        const float d = __fdiv_rn(amax, 127.0f);
        const float id = (d != 0.0f) ? __fdiv_rn(1.0f, d) : 0.0f;
        int sum = 0;
        uint32_t packed[8];
#pragma unroll
        for (int v = 0; v < 8; ++v) {
            uint32_t word = 0;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                float q = roundf(__fmul_rn(xh[4 * v + c], id));
                q = fminf(fmaxf(q, -127.0f), 127.0f);
                const int qi = (int)q;
                sum += qi;
                word |= ((uint32_t)(qi & 0xFF)) << (8 * c);
            }
            packed[v] = word;
        }
        uint4 *dst = reinterpret_cast<uint4 *>(qs + (size_t)blockIdx.x * K + 32 * b);
        dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
        dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
        const size_t o = (size_t)blockIdx.x * nblk + b;
        dq[o] = __float2half_rn(d);
        sq[o] = __float2half_rn(__fmul_rn(d, (float)sum));
    }
}

}  // namespace

cudaError_t launch_rmsnorm_q8_1(const float *x, const float *gamma, int B, int K,
                                float eps, zq_q8_1 out, cudaStream_t st)
{
    rmsnorm_q8_1_kernel<<<B, kThreads, 0, st>>>(
        x, gamma, K, eps, out.qs, reinterpret_cast<__half *>(out.d),
        reinterpret_cast<__half *>(out.s));
    return cudaGetLastError();
}

}  // namespace zq
