// q4k_dequant.cu -- Q4_K weights (and Q8_1 activations) dequantised to
// binary16, the first step of a dequantise-then-GEMM prefill (MIInfer README, "Current phase": Q4_K
// dequantised to 16-bit weights ahead of a dense GEMM, its best prefill lever).
//
// The library's own prefill keeps the weights in Q4_K and converts them tile
// by tile inside the tensor-core kernel; this kernel exists so that the
// dequantise-then-GEMM design can be measured beside it.  Per weight, in
// fp32: a = d*sc and b = dmin*m (both exact), w = a*q - b (a*q exact, one
// rounding), then w rounded to binary16.  One thread decodes one 32-byte
// nibble group (64 weights) of one super-block of one row.  HBM roofline:
// reads N*K*0.5625 bytes, writes N*K*2.
#include "zq_internal.cuh"

namespace zq {
namespace {

__global__ void q4k_dequant_f16_kernel(const uint8_t *__restrict__ W, int nb, size_t groups, int K,
                                       __half *__restrict__ out)
{
    const size_t t = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= groups) return;
    const int g = (int)(t & 3);
    const size_t rb = t >> 2;   // row * nb + super-block
    const int b = (int)(rb % (size_t)nb);
    const size_t n = rb / (size_t)nb;
    const uint8_t *blk = W + rb * kQ4KBlockBytes;
    const uint4 hdr = ld_stream_u4(blk);
    const uint4 n0 = ld_stream_u4(blk + 16 + 32 * g);
    const uint4 n1 = ld_stream_u4(blk + 32 + 32 * g);
    const float2 dm = __half22float2(*reinterpret_cast<const __half2 *>(&hdr.x));
    uint32_t sc0, m0, sc1, m1;
    q4k_scale_min(hdr.y, hdr.z, hdr.w, 2 * g, sc0, m0);
    q4k_scale_min(hdr.y, hdr.z, hdr.w, 2 * g + 1, sc1, m1);
    const float a0 = __fmul_rn(dm.x, (float)sc0), b0 = __fmul_rn(dm.y, (float)m0);
    const float a1 = __fmul_rn(dm.x, (float)sc1), b1 = __fmul_rn(dm.y, (float)m1);
    const uint32_t wv[8] = {n0.x, n0.y, n0.z, n0.w, n1.x, n1.y, n1.z, n1.w};
    uint32_t lo[16], hi[16];
#pragma unroll
    for (int v = 0; v < 8; ++v) {
#pragma unroll
        for (int c = 0; c < 4; c += 2) {
            const uint32_t b0w = (wv[v] >> (8 * c)) & 0xFFu, b1w = (wv[v] >> (8 * c + 8)) & 0xFFu;
            const __half2 l = __floats2half2_rn(__fsub_rn(__fmul_rn(a0, (float)(b0w & 15u)), b0),
                                                __fsub_rn(__fmul_rn(a0, (float)(b1w & 15u)), b0));
            const __half2 h = __floats2half2_rn(__fsub_rn(__fmul_rn(a1, (float)(b0w >> 4)), b1),
                                                __fsub_rn(__fmul_rn(a1, (float)(b1w >> 4)), b1));
            lo[2 * v + c / 2] = *reinterpret_cast<const uint32_t *>(&l);
            hi[2 * v + c / 2] = *reinterpret_cast<const uint32_t *>(&h);
        }
    }
    // sub-block 2g: weights 64g .. 64g+31; sub-block 2g+1: 64g+32 .. 64g+63
    uint4 *dst = reinterpret_cast<uint4 *>(out + n * (size_t)K + 256 * (size_t)b + 64 * g);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        dst[i] = make_uint4(lo[4 * i], lo[4 * i + 1], lo[4 * i + 2], lo[4 * i + 3]);
        dst[4 + i] = make_uint4(hi[4 * i], hi[4 * i + 1], hi[4 * i + 2], hi[4 * i + 3]);
    }
}

// Q8_1 activations dequantised to binary16, x = q8 * d8 (exact in fp32,
// then one rounding to binary16, nearest even): eight codes per thread.
__global__ void q8_1_dequant_f16_kernel(const int8_t *__restrict__ qs, const __half *__restrict__ d, size_t groups,
                                        __half *__restrict__ out)
{
    const size_t t = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= groups) return;
    const uint2 q = *reinterpret_cast<const uint2 *>(qs + 8 * t);
    const float d8 = __half2float(d[t >> 2]);   // four groups of eight per Q8_1 block
    const uint32_t w[2] = {q.x, q.y};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int8_t c0 = (int8_t)((w[i >> 1] >> (16 * (i & 1))) & 0xFFu);
        const int8_t c1 = (int8_t)((w[i >> 1] >> (16 * (i & 1) + 8)) & 0xFFu);
        const __half2 h = __floats2half2_rn(__fmul_rn((float)c0, d8), __fmul_rn((float)c1, d8));
        o[i] = *reinterpret_cast<const uint32_t *>(&h);
    }
    *reinterpret_cast<uint4 *>(out + 8 * t) = make_uint4(o[0], o[1], o[2], o[3]);
}

}  // namespace

cudaError_t launch_q8_1_dequant_f16(zq_q8_1 a, int B, int K, void *out, cudaStream_t st)
{
    const size_t groups = (size_t)B * K / 8;
    if (groups == 0) return cudaSuccess;
    q8_1_dequant_f16_kernel<<<(unsigned)((groups + 255) / 256), 256, 0, st>>>(
        a.qs, reinterpret_cast<const __half *>(a.d), groups, static_cast<__half *>(out));
    return cudaGetLastError();
}

cudaError_t launch_q4k_dequant_f16(const void *W, int N, int K, void *out, cudaStream_t st)
{
    const int nb = K / 256;
    const size_t groups = (size_t)N * nb * 4;
    q4k_dequant_f16_kernel<<<(unsigned)((groups + 255) / 256), 256, 0, st>>>(
        static_cast<const uint8_t *>(W), nb, groups, K, static_cast<__half *>(out));
    return cudaGetLastError();
}

}  // namespace zq
