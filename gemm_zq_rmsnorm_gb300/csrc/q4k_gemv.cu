// q4k_gemv.cu -- Q4_K x Q8_1 mat-vec on the integer dot-product units.
//
// MIInfer README, "Status": Q4_K x Q8_1 MMVQ-style projections (FFN down,
// shared gate/up), Q4_K metadata staging (+38 % decode) and the packed int8
// dot4 projection path (+9.6/10.0 %).  ZINC docs "ROCm backend", "Build and
// verify": paired Q4 projections for gate/up.
//
// Decode (B = 1) is bound by HBM: every weight byte is read exactly once
// (N*K*144/256 bytes), the activation row (K*1.125 bytes) is read from L1/L2
// by every warp.  The kernel therefore streams the weights with coalesced
// 16-byte non-allocating loads and keeps several super-blocks per lane in
// flight, decodes nibbles and 6-bit scales in registers and does the 32-wide
// sub-block sums with dp4a.
//
// Lane mapping inside a warp (32 lanes, 4 consecutive super-blocks of one
// row per step, 576 contiguous bytes):
//   g = lane / 8  selects the super-block b = 4*step + g;
//   i = lane % 8  selects the 16 nibble bytes 16*i .. 16*i+15 of that block,
//                 i.e. positions 16*(i%2) .. +15 of sub-blocks j0 = 2*(i/2)
//                 (low nibbles) and j1 = j0 + 1 (high nibbles);
//   every lane also reads the block's 16-byte header (d, dmin, 12 scale
//   bytes); the eight lanes of a block share that load.
// Each lane accumulates d*(sc0*d8_0*I0 + sc1*d8_1*I1) - dmin*m*s8 for its
// half sub-blocks (the min term of sub-block j0 on the even lane, j1 on the
// odd lane) and the warp reduces once per row at the end.
//
// The same kernel, with NT tokens per warp, serves any B (each warp streams
// one weight row once for NT tokens), and with ISUMS exports the exact
// sub-block integer sums for testing.
#include "zq_internal.cuh"

namespace zq {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;  // super-block steps in flight per lane

struct LaneBlock {
    uint4 hdr;  // d | dmin, S[0..3], S[4..7], S[8..11]
    uint4 q;    // 16 nibble bytes
};

template <int NT, bool PAIR, bool ISUMS>
__global__ void __launch_bounds__(kThreads)
q4k_mv_kernel(const uint8_t *__restrict__ W, const uint8_t *__restrict__ W2, int N, int K,
              const int8_t *__restrict__ qs, const __half *__restrict__ dq,
              const __half *__restrict__ sq, int B, float *__restrict__ y,
              float *__restrict__ y2, int32_t *__restrict__ isums)
{
    const int lane = threadIdx.x & 31;
    const int g = lane >> 3;
    const int i = lane & 7;
    const int j0 = (i >> 1) * 2;
    const int h = i & 1;
    const int nb = K >> 8;
    const int nsub = K >> 5;
    const size_t row_bytes = (size_t)nb * kQ4KBlockBytes;
    const int ngroups = (B + NT - 1) / NT;
    const long long units = (long long)N * ngroups;
    const int warps_total = gridDim.x * (kThreads / 32);

    for (long long u = (long long)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); u < units;
         u += warps_total) {
        const int n = (int)(u % N);
        const int t0 = (int)(u / N) * NT;
        const uint8_t *row = W + (size_t)n * row_bytes;
        const uint8_t *row2 = PAIR ? W2 + (size_t)n * row_bytes : nullptr;
        float acc[NT], acc2[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) acc[t] = acc2[t] = 0.0f;

        for (int b0 = 0; b0 < nb; b0 += 4 * kUnroll) {
            LaneBlock lb[kUnroll], lb2[kUnroll];
#pragma unroll
            for (int s = 0; s < kUnroll; ++s) {
                const int b = b0 + 4 * s + g;
                if (b < nb) {
                    const uint8_t *blk = row + (size_t)b * kQ4KBlockBytes;
                    lb[s].hdr = ld_stream_u4(blk);
                    lb[s].q = ld_stream_u4(blk + 16 + 16 * i);
                    if (PAIR) {
                        const uint8_t *blk2 = row2 + (size_t)b * kQ4KBlockBytes;
                        lb2[s].hdr = ld_stream_u4(blk2);
                        lb2[s].q = ld_stream_u4(blk2 + 16 + 16 * i);
                    }
                }
            }
#pragma unroll
            for (int s = 0; s < kUnroll; ++s) {
                const int b = b0 + 4 * s + g;
                if (b >= nb) continue;
                const int sub0 = 8 * b + j0;  // sub-block index of j0 in the row
                const int k0 = 32 * sub0 + 16 * h;
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    const int tok = t0 + t;
                    if (tok >= B) break;
                    const int8_t *arow = qs + (size_t)tok * K;
                    const uint4 a0 = ld_cached_u4(arow + k0);
                    const uint4 a1 = ld_cached_u4(arow + k0 + 32);
                    const float d80 = __half2float(dq[(size_t)tok * nsub + sub0]);
                    const float d81 = __half2float(dq[(size_t)tok * nsub + sub0 + 1]);
                    const float s8 = __half2float(sq[(size_t)tok * nsub + sub0 + h]);
#pragma unroll
                    for (int w = 0; w < (PAIR ? 2 : 1); ++w) {
                        const LaneBlock &L = (w == 0) ? lb[s] : lb2[s];
                        const uint32_t q0 = L.q.x, q1 = L.q.y, q2 = L.q.z, q3 = L.q.w;
                        int I0 = 0, I1 = 0;
                        I0 = __dp4a((int)(q0 & 0x0F0F0F0Fu), (int)a0.x, I0);
                        I0 = __dp4a((int)(q1 & 0x0F0F0F0Fu), (int)a0.y, I0);
                        I0 = __dp4a((int)(q2 & 0x0F0F0F0Fu), (int)a0.z, I0);
                        I0 = __dp4a((int)(q3 & 0x0F0F0F0Fu), (int)a0.w, I0);
                        I1 = __dp4a((int)((q0 >> 4) & 0x0F0F0F0Fu), (int)a1.x, I1);
                        I1 = __dp4a((int)((q1 >> 4) & 0x0F0F0F0Fu), (int)a1.y, I1);
                        I1 = __dp4a((int)((q2 >> 4) & 0x0F0F0F0Fu), (int)a1.z, I1);
                        I1 = __dp4a((int)((q3 >> 4) & 0x0F0F0F0Fu), (int)a1.w, I1);
                        if (ISUMS) {
                            // join the two half sub-blocks held by lanes i, i^1
                            // (the 8 lanes of one super-block agree on validity)
                            const unsigned gm = 0xFFu << (8 * g);
                            const int J0 = I0 + __shfl_xor_sync(gm, I0, 1);
                            const int J1 = I1 + __shfl_xor_sync(gm, I1, 1);
                            int32_t *dst = isums + ((size_t)tok * N + n) * nsub + sub0;
                            dst[h] = h ? J1 : J0;
                            continue;
                        }
                        uint32_t sc0, m0, sc1, m1;
                        q4k_scale_min(L.hdr.y, L.hdr.z, L.hdr.w, j0, sc0, m0);
                        q4k_scale_min(L.hdr.y, L.hdr.z, L.hdr.w, j0 + 1, sc1, m1);
                        const float d = __half2float(__ushort_as_half((uint16_t)(L.hdr.x & 0xFFFFu)));
                        const float dmin = __half2float(__ushort_as_half((uint16_t)(L.hdr.x >> 16)));
                        const float main = fmaf((float)sc1 * d81, (float)I1, (float)sc0 * d80 * (float)I0);
                        const float mterm = (float)(h ? m1 : m0) * s8;
                        float &A = (w == 0) ? acc[t] : acc2[t];
                        A = fmaf(d, main, A);
                        A = fmaf(-dmin, mterm, A);
                    }
                }
            }
        }
        if (ISUMS) continue;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            float v = acc[t], v2 = acc2[t];
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) {
                v += __shfl_xor_sync(0xffffffffu, v, off);
                if (PAIR) v2 += __shfl_xor_sync(0xffffffffu, v2, off);
            }
            const int tok = t0 + t;
            if (lane == 0 && tok < B) {
                y[(size_t)tok * N + n] = v;
                if (PAIR) y2[(size_t)tok * N + n] = v2;
            }
        }
    }
}

template <int NT, bool PAIR, bool ISUMS>
cudaError_t launch_mv(const void *W, const void *W2, int N, int K, zq_q8_1 a, int B, float *y,
                      float *y2, int32_t *isums, cudaStream_t st)
{
    const long long units = (long long)N * ((B + NT - 1) / NT);
    const long long want = (units + (kThreads / 32) - 1) / (kThreads / 32);
    const long long cap = (long long)num_sms() * 8;
    const int grid = (int)(want < cap ? want : cap);
    q4k_mv_kernel<NT, PAIR, ISUMS><<<grid, kThreads, 0, st>>>(
        static_cast<const uint8_t *>(W), static_cast<const uint8_t *>(W2), N, K, a.qs,
        reinterpret_cast<const __half *>(a.d), reinterpret_cast<const __half *>(a.s), B, y, y2,
        isums);
    return cudaGetLastError();
}

}  // namespace

// W2 != nullptr selects the paired kernel (B must be 1); isums != nullptr
// selects the integer-sum export.
cudaError_t launch_gemv(const void *W, const void *W2, int N, int K, zq_q8_1 a, int B, float *y,
                        float *y2, int32_t *isums, cudaStream_t st)
{
    if (isums) return launch_mv<1, false, true>(W, nullptr, N, K, a, B, nullptr, nullptr, isums, st);
    if (W2) return launch_mv<1, true, false>(W, W2, N, K, a, B, y, y2, nullptr, st);
    if (B == 1) return launch_mv<1, false, false>(W, nullptr, N, K, a, B, y, nullptr, nullptr, st);
    return launch_mv<4, false, false>(W, nullptr, N, K, a, B, y, nullptr, nullptr, st);
}

}  // namespace zq
