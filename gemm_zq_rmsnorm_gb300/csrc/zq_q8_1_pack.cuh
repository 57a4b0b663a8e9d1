// zq_q8_1_pack.cuh -- packing of one normalised 32-value block into Q8_1 and
// the canonical RMSNorm pieces, shared by the RMSNorm+Q8_1 kernels and the
// decode mat-vec that normalises its input itself, so both produce the same
// bytes.
//
// ZINC docs "ROCm backend", "Build and verify": Q8 activation packing for the
// Q4_K projections, fused with RMS normalisation.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace zq {

struct Q8Block {
    uint4 q0, q1;   // the 32 codes
    __half d, s;    // binary16 scale and scaled code sum
};

// d = amax/127 in fp32, q = round-half-away(xh * (1/d)) clamped to +-127,
// s = d * sum(q); d and s rounded to binary16 (nearest even).
__device__ __forceinline__ Q8Block q8_1_pack(const float (&xh)[32])
{
    float amax = 0.0f;
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
    Q8Block o;
    o.q0 = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    o.q1 = make_uint4(packed[4], packed[5], packed[6], packed[7]);
    o.d = __float2half_rn(d);
    o.s = __float2half_rn(__fmul_rn(d, (float)sum));
    return o;
}

// The batched projection's power-of-two scale for one token's activations:
// k = 0 when 127 * max|d8| fits binary16 (<= 65504), else the exponent e of
// 127 * max|d8| / 65504 = f * 2^e with f in [0.5, 1), so every |q8 * d8| *
// 2^-k stays within binary16 range.  Read from the quotient's exponent field
// (the quotient is >= 1, a normal number).
__device__ __forceinline__ int split_scale_exp(float dmax)
{
    const float bound = 127.0f * dmax;
    if (!(bound > 65504.0f)) return 0;
    return (int)((__float_as_uint(__fdiv_rn(bound, 65504.0f)) >> 23) & 0xFFu) - 126;
}

// 2^e for e in [-126, 127], built from its exponent field
__device__ __forceinline__ float pow2_exact(int e) { return __int_as_float((127 + e) << 23); }

// p_b of the canonical order: a fused multiply-add chain over the squares of
// one 32-value block, in index order, from +0.
__device__ __forceinline__ float block_sumsq(const float *xb)
{
    const float4 *p = reinterpret_cast<const float4 *>(xb);
    float part = 0.0f;
#pragma unroll
    for (int v = 0; v < 8; ++v) {
        const float4 f = __ldg(p + v);
        part = __fmaf_rn(f.x, f.x, part);
        part = __fmaf_rn(f.y, f.y, part);
        part = __fmaf_rn(f.z, f.z, part);
        part = __fmaf_rn(f.w, f.w, part);
    }
    return part;
}

// r = 1 / sqrt(ss / K + eps), each step one IEEE fp32 operation
__device__ __forceinline__ float rms_scale(float ss, int K, float eps)
{
    const float mean = __fdiv_rn(ss, (float)K);
    return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, eps)));
}

// xh = (x * r) * gamma for one block, two roundings per value
__device__ __forceinline__ void block_normalise(const float *xb, const float *gb, float r, float (&xh)[32])
{
    const float4 *p = reinterpret_cast<const float4 *>(xb);
    const float4 *g = reinterpret_cast<const float4 *>(gb);
#pragma unroll
    for (int v = 0; v < 8; ++v) {
        const float4 f = __ldg(p + v);
        const float4 w = __ldg(g + v);
        xh[4 * v + 0] = __fmul_rn(__fmul_rn(f.x, r), w.x);
        xh[4 * v + 1] = __fmul_rn(__fmul_rn(f.y, r), w.y);
        xh[4 * v + 2] = __fmul_rn(__fmul_rn(f.z, r), w.z);
        xh[4 * v + 3] = __fmul_rn(__fmul_rn(f.w, r), w.w);
    }
}

// SiLU(gate) * up in the library's fp32 steps (every implementation that
// follows them gets the same value, hence the same Q8_1 codes; MIInfer
// README, "Current phase": SiLU(gate)*up feeding the down projection):
//   exp32(a): a clamped to [-86, 88]; k = rint(a * log2 e);
//     r = fma(-k, ln2_hi, a); r = fma(-k, ln2_lo, r)  (ln 2 split in two, the
//     high part exact in 16 bits); p = Horner sum of r^n/n!, n <= 7, with fma;
//     result p * 2^k (exact);
//   silu(g) = g / (1 + exp32(-g));  h = silu(g) * u.
__device__ __forceinline__ float exp32(float a)
{
    a = fminf(fmaxf(a, -86.0f), 88.0f);
    const float kf = rintf(__fmul_rn(a, 0x1.715476p+0f));
    float r = __fmaf_rn(-kf, 0x1.62e4p-1f, a);
    r = __fmaf_rn(-kf, 0x1.7f7d1cp-20f, r);
    float p = 0x1.a01a02p-13f;
    p = __fmaf_rn(p, r, 0x1.6c16c2p-10f);
    p = __fmaf_rn(p, r, 0x1.111112p-7f);
    p = __fmaf_rn(p, r, 0x1.555556p-5f);
    p = __fmaf_rn(p, r, 0x1.555556p-3f);
    p = __fmaf_rn(p, r, 0.5f);
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    return __fmul_rn(p, __int_as_float(((int)kf + 127) << 23));
}

__device__ __forceinline__ float silu_mul(float g, float u)
{
    return __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, exp32(-g))), u);
}

}  // namespace zq
