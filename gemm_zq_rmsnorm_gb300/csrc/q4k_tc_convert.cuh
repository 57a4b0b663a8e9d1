// q4k_tc_convert.cuh -- Q4_K weights converted for the binary16 tensor-core
// MMAs of the batched projection kernels (CTA-pair prefill and chunk
// kernels), and the per-super-block fold of their accumulators.
//
// The projection is
//   y[t][n] = sum_b d_b[n] * ( sum_{k in b} x'[t][k] * w[n][k]
//                              - (dmin_b[n] / d_b[n]) * sum_j m_j[n] * s8[t][bj] ),
// x' = q8 * d8 (split into exact binary16 hi + lo), w = sc_j * q4 (exact in
// binary16).  The min term enters the same accumulator through one more
// K = 16 MMA whose A operand holds -(dmin/d) * m_j as binary16 hi and lo
// parts and whose B operand holds the token's eight s8 values twice.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "zq_async.cuh"
#include "zq_internal.cuh"
#include "zq_tc.cuh"
#include "zq_tc_common.cuh"

namespace zq {
namespace {

// Per weight row and super-block: a power of two 2^-e applied to w = sc*q
// (0 when d = 0), the ratio r whose binary16 parts carry the min term
// (-r * m_j), and the fold factor of the accumulator, so that
// fold * (wmul * w * x' - r * m * s8) = d * w * x' - dmin * m * s8.
// e comes from the binary16 exponents alone (integer arithmetic, identical in
// the converters and the epilogue): it keeps |r * m| < 2^14, so the parts of
// the min operand stay in binary16 range; wmul * w stays exact while e <= 24
// (dmin / d below 2^31).
struct Fold {
    float wmul, fold;
    int e;
};

// floor(log2 |v|) of a non-zero binary16 magnitude (subnormals included)
__device__ __forceinline__ int f16_ilog2(uint32_t h)
{
    const uint32_t E = (h >> 10) & 31u, M = h & 1023u;
    return E ? (int)E - 15 : -24 + 31 - __clz((int)M);
}

__device__ __forceinline__ Fold fold_of(uint32_t d_dmin)
{
    const uint32_t hd = d_dmin & 0x7FFFu, hm = (d_dmin >> 16) & 0x7FFFu;
    int e = 0;
    if (hm) e = max(0, f16_ilog2(hm) - (hd ? f16_ilog2(hd) : 0) - 7);
    Fold f;
    f.e = e;
    f.wmul = hd ? ldexpf(1.0f, -e) : 0.0f;
    const float d = __half2float(__ushort_as_half((unsigned short)(d_dmin & 0xFFFFu)));
    f.fold = ldexpf(hd ? d : 1.0f, e);
    return f;
}

// r * 2^-e: dmin / d (dmin itself when d = 0), scaled
__device__ __forceinline__ float ratio_of(uint32_t d_dmin, int e)
{
    const float d = __half2float(__ushort_as_half((unsigned short)(d_dmin & 0xFFFFu)));
    const float dm = __half2float(__ushort_as_half((unsigned short)(d_dmin >> 16)));
    return ldexpf((d_dmin & 0x7FFFu) ? dm / d : dm, -e);
}

// Converts stage I (sub-blocks 2I, 2I+1) of one weight row and stores it in
// the row's lane of a tensor-memory A slot at column address `col`: binary16
// pairs in K order, the low nibbles (sub-block 2I) in columns 0..15, the
// high nibbles (2I+1) in 16..31; for I = 3 also the row's min operand
// (-r * m_j as binary16 hi, then lo) in its 32-byte-swizzled shared-memory
// row `mrow`.
template <int I>
__device__ __forceinline__ void convert_one(const uint8_t *raw, uint32_t col, uint8_t *mrow, int r)
{
    const uint4 hdr = *reinterpret_cast<const uint4 *>(raw);
    const uint4 n0 = *reinterpret_cast<const uint4 *>(raw + 16 + 32 * I);
    const uint4 n1 = *reinterpret_cast<const uint4 *>(raw + 32 + 32 * I);
    const Fold f = fold_of(hdr.x);
    const uint32_t wv[8] = {n0.x, n0.y, n0.z, n0.w, n1.x, n1.y, n1.z, n1.w};
#pragma unroll
    for (int hi = 0; hi < 2; ++hi) {
        uint32_t sc, md;
        q4k_scale_min(hdr.y, hdr.z, hdr.w, 2 * I + hi, sc, md);
        const float scf = (float)sc * f.wmul;
        const __half2 s2 = __float2half2_rn(hi ? scf * 0.0625f : scf);
        const __half2 o2 = __float2half2_rn(hi ? -64.0f * scf : -1024.0f * scf);
        const uint32_t m = hi ? 0x00F000F0u : 0x000F000Fu;
        uint32_t o[16];
#pragma unroll
        for (int c = 0; c < 8; ++c) {   // nibble bytes 4c..4c+3 -> columns 2c, 2c+1
            const uint32_t p0 = (__byte_perm(wv[c], 0, 0x4140) & m) | 0x64006400u;   // bytes 0, 1
            const uint32_t p1 = (__byte_perm(wv[c], 0, 0x4342) & m) | 0x64006400u;   // bytes 2, 3
            o[2 * c] = h2_bits(__hfma2(*reinterpret_cast<const __half2 *>(&p0), s2, o2));
            o[2 * c + 1] = h2_bits(__hfma2(*reinterpret_cast<const __half2 *>(&p1), s2, o2));
        }
        tmem_st16(col + 16u * hi, o);
    }
    if (I == 3) {
        const float rr = ratio_of(hdr.x, f.e);
        uint32_t hv[4], lv[4];
#pragma unroll
        for (int j = 0; j < 8; j += 2) {
            uint32_t m0v, m1v, scd;
            q4k_scale_min(hdr.y, hdr.z, hdr.w, j, scd, m0v);
            q4k_scale_min(hdr.y, hdr.z, hdr.w, j + 1, scd, m1v);
            const float v0 = -rr * (float)m0v, v1 = -rr * (float)m1v;
            const __half2 hh = __floats2half2_rn(v0, v1);
            const float2 hb = __half22float2(hh);
            hv[j >> 1] = h2_bits(hh);
            lv[j >> 1] = h2_bits(__floats2half2_rn(v0 - hb.x, v1 - hb.y));
        }
        const int s32 = (r >> 2) & 1;
        *reinterpret_cast<uint4 *>(mrow + ((0 ^ s32) << 4)) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
        *reinterpret_cast<uint4 *>(mrow + ((1 ^ s32) << 4)) = make_uint4(lv[0], lv[1], lv[2], lv[3]);
        fence_async_smem();   // the min MMA reads this row through the async proxy
    }
}

__device__ __forceinline__ void fma2(float &c0, float &c1, float a, float b0, float b1)
{
    asm("{\n\t.reg .b64 ra, rb, rc;\n\t"
        "mov.b64 ra, {%2, %2};\n\tmov.b64 rb, {%3, %4};\n\tmov.b64 rc, {%0, %1};\n\t"
        "fma.rn.f32x2 rc, ra, rb, rc;\n\tmov.b64 {%0, %1}, rc;\n\t}"
        : "+f"(c0), "+f"(c1)
        : "f"(a), "f"(b0), "f"(b1));
}

__device__ __forceinline__ uint32_t ld_nc_u32(const void *p)
{
    uint32_t v;
    asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

}  // namespace
}  // namespace zq
