// q4k_gemm_tc.cu -- the batched Q4_K x Q8_1 projection's dispatch and the
// pieces its tensor-core kernels share: the split of the Q8_1 activations
// into exact binary16 hi + lo parts (and the scaled s8 operand), the split-K
// reduction, tensor maps, split counts and the workspace layout.
//
// MIInfer README, "Current phase": token-batched chunk projections and
// tensor-core prefill.  B >= 17 runs the CTA-pair kernel (q4k_gemm_2sm.cu),
// 5 <= B <= 16 the chunk kernel (q4k_gemm_chunk.cu); both read the
// activations as x' = q8 * d8 split into binary16 hi + lo, so that every
// product with a weight code sc * q4 is exact.
#include <cuda.h>

#include "zq_internal.cuh"
#include "zq_q8_1_pack.cuh"
#include "zq_tc.cuh"
#include "zq_tc_common.cuh"

namespace zq {
namespace {

// CTA (t, c): token t's super-blocks c*sbc .. (c+1)*sbc - 1, x' = q8 * d8
// split into binary16 hi + lo.  The token's codes are scaled by 2^-k, k >= 0
// the least that keeps 127 * max d8 within binary16 range (every CTA of the
// token finds the same maximum over all its d8), and tscale[t] = 2^k.
constexpr int kSplitThreads = 256;

__global__ void __launch_bounds__(kSplitThreads)
q8_split_kernel(const int8_t *__restrict__ qs, const __half *__restrict__ d8, const __half *__restrict__ s8, int K,
                int sbc, __half *__restrict__ hi, __half *__restrict__ lo, float *__restrict__ tscale,
                __half *__restrict__ s8x)
{
    __shared__ float red[kSplitThreads / 32];
    const int t = blockIdx.x;
    const int nblk = K >> 5;
    const __half *dt = d8 + (size_t)t * nblk;
    float m = 0.0f;
    for (int j = threadIdx.x; j < nblk; j += kSplitThreads) m = fmaxf(m, fabsf(__half2float(dt[j])));
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    m = red[0];
#pragma unroll
    for (int w = 1; w < kSplitThreads / 32; ++w) m = fmaxf(m, red[w]);
    const int k = split_scale_exp(m);   // 127 * m bounds every |x'| of the token
    const float down = pow2_exact(-k);
    if (threadIdx.x == 0 && blockIdx.y == 0) tscale[t] = pow2_exact(k);
    const int8_t *qt = qs + (size_t)t * K;
    const int sb0 = blockIdx.y * sbc, sb1 = min(K >> 8, sb0 + sbc);   // this CTA's super-blocks
    for (int g = 16 * sb0 + threadIdx.x; g < 16 * sb1; g += kSplitThreads) {
        const int4 v = __ldg(reinterpret_cast<const int4 *>(qt) + g);
        const float dv = __half2float(dt[g >> 1]) * down;
        const int w[4] = {v.x, v.y, v.z, v.w};
        uint32_t oh[8], ol[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int x = w[i >> 1];
            float a[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) a[h] = (float)(int8_t)((x >> (16 * (i & 1) + 8 * h)) & 0xFF) * dv;
            const __half2 vh = __floats2half2_rn(a[0], a[1]);
            const float2 back = __half22float2(vh);
            oh[i] = h2_bits(vh);
            ol[i] = h2_bits(__floats2half2_rn(a[0] - back.x, a[1] - back.y));
        }
        uint4 *dh = reinterpret_cast<uint4 *>(hi + (size_t)t * K) + 2 * g;
        uint4 *dl = reinterpret_cast<uint4 *>(lo + (size_t)t * K) + 2 * g;
        dh[0] = make_uint4(oh[0], oh[1], oh[2], oh[3]);
        dh[1] = make_uint4(oh[4], oh[5], oh[6], oh[7]);
        dl[0] = make_uint4(ol[0], ol[1], ol[2], ol[3]);
        dl[1] = make_uint4(ol[4], ol[5], ol[6], ol[7]);
    }
    if (s8x) {
        // per super-block g: its eight s8 values scaled like the codes,
        // twice (the B operand of the pair kernel's min-term MMA)
        const uint4 *st = reinterpret_cast<const uint4 *>(s8 + (size_t)t * nblk);
        uint4 *dx = reinterpret_cast<uint4 *>(s8x + (size_t)t * (K >> 4));
        for (int g = sb0 + threadIdx.x; g < sb1; g += kSplitThreads) {
            const uint4 v = __ldg(st + g);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            uint32_t o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[i]));
                o[i] = h2_bits(__floats2half2_rn(f.x * down, f.y * down));
            }
            dx[2 * g] = make_uint4(o[0], o[1], o[2], o[3]);
            dx[2 * g + 1] = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

// q8 codes -> fp16 (exact), 16 per thread
__global__ void q8_to_f16_kernel(const int8_t *__restrict__ qs, __half *__restrict__ out, size_t n16)
{
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n16) return;
    const int4 v = __ldg(reinterpret_cast<const int4 *>(qs) + i);
    const int w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int x = w[k];
        o[2 * k] = h2_bits(__floats2half2_rn((float)(int8_t)(x & 0xFF), (float)(int8_t)((x >> 8) & 0xFF)));
        o[2 * k + 1] = h2_bits(__floats2half2_rn((float)(int8_t)((x >> 16) & 0xFF), (float)(int8_t)(x >> 24)));
    }
    uint4 *dst = reinterpret_cast<uint4 *>(out) + 2 * i;
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
}

// y = sum over the splits of the partial products, in split order.  Thread i
// adds group i of four consecutive outputs; the last group of a ragged B * N
// (n % 4 != 0) is added element by element.
__global__ void splitk_reduce_kernel(const float *__restrict__ part, int splits, size_t n, size_t stride,
                                     float *__restrict__ y)
{
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    const size_t e0 = 4 * i;
    if (e0 >= n) return;
    if (e0 + 4 <= n) {
        float4 a = __ldg(reinterpret_cast<const float4 *>(part + e0));
        for (int s = 1; s < splits; ++s) {
            const float4 b = __ldg(reinterpret_cast<const float4 *>(part + (size_t)s * stride + e0));
            a.x += b.x;
            a.y += b.y;
            a.z += b.z;
            a.w += b.w;
        }
        *reinterpret_cast<float4 *>(y + e0) = a;
        return;
    }
    for (size_t e = e0; e < n; ++e) {
        float a = __ldg(part + e);
        for (int s = 1; s < splits; ++s) a += __ldg(part + (size_t)s * stride + e);
        y[e] = a;
    }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

size_t g_attr_bytes[64];

}  // namespace

// workspace layout: hi [B][K] fp16 | lo [B][K] fp16 | tscale [B] fp32 |
// (B >= 17) s8x [B][K/16] fp16 | partial sums [splits][split_stride(B, N)]
// fp32 (when splits > 1); each region padded to 256 bytes
size_t split_bytes(int K, int B) { return (size_t)B * K * sizeof(__half); }
size_t tscale_bytes(int B) { return ((size_t)B * sizeof(float) + 255) & ~(size_t)255; }
size_t s8x_bytes(int K, int B) { return B > 1 ? (((size_t)B * (K / 16) * sizeof(__half) + 255) & ~(size_t)255) : 0; }

cudaError_t launch_q8_split(zq_q8_1 a, int K, int B, __half *hi, __half *lo, float *tscale, __half *s8x,
                            cudaStream_t st)
{
    // few tokens: split each token's K over several CTAs (two or more CTAs per SM in all)
    const int nb = K / 256;
    int chunks = (2 * num_sms() + B - 1) / B;
    chunks = chunks < 1 ? 1 : (chunks > nb ? nb : chunks);
    const int sbc = (nb + chunks - 1) / chunks;
    chunks = (nb + sbc - 1) / sbc;
    q8_split_kernel<<<dim3(B, chunks), kSplitThreads, 0, st>>>(a.qs, reinterpret_cast<const __half *>(a.d),
                                                               reinterpret_cast<const __half *>(a.s), K, sbc, hi, lo,
                                                               tscale, s8x);
    return cudaGetLastError();
}

cudaError_t launch_splitk_reduce(const float *part, int splits, size_t n, float *y, cudaStream_t st)
{
    const size_t groups = (n + 3) / 4;
    const size_t stride = (n + 3) & ~(size_t)3;
    splitk_reduce_kernel<<<(unsigned)((groups + 255) / 256), 256, 0, st>>>(part, splits, n, stride, y);
    return cudaGetLastError();
}

cudaError_t make_tmap_2d(CUtensorMap *m, CUtensorMapDataType dt, uint32_t esize, const void *base, uint64_t cols,
                         uint64_t rows, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle sw)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * esize};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t launch_q8_to_f16(const int8_t *qs, __half *out, size_t n, cudaStream_t st)
{
    const size_t n16 = n / 16;
    if (n16 == 0) return cudaSuccess;
    q8_to_f16_kernel<<<(unsigned)((n16 + 255) / 256), 256, 0, st>>>(qs, out, n16);
    return cudaGetLastError();
}

int gemm_splits(int B, int N, int K, bool allow_split)
{
    if (!allow_split || B <= kSmallMaxB) return 1;
    return choose_splits_pair(B, N, K, num_sms());
}

// Partial-sum bytes: split-K slices (B > 16) or the pieces of tiles that
// straddle the chunk kernel's ranges (B <= 16); none without splitting.
static size_t part_bytes(int N, int K, int B, bool allow_split)
{
    if (!allow_split) return 0;
    if (B <= kSmallMaxB) return chunk_part_bytes(N, K, B);
    const int sp = gemm_splits(B, N, K, true);
    return sp > 1 ? (size_t)sp * split_stride(B, N) * sizeof(float) : 0;
}

size_t gemm_tc_workspace_bytes(int N, int K, int B, bool allow_split)
{
    if (B <= 1) return 0;
    return 2 * split_bytes(K, B) + tscale_bytes(B) + s8x_bytes(K, B) + part_bytes(N, K, B, allow_split);
}

TcWorkspace tc_workspace(void *ws, int K, int B)
{
    uint8_t *w8 = static_cast<uint8_t *>(ws);
    TcWorkspace w;
    w.hi = reinterpret_cast<__half *>(w8);
    w.lo = reinterpret_cast<__half *>(w8 + split_bytes(K, B));
    w.tscale = reinterpret_cast<float *>(w8 + 2 * split_bytes(K, B));
    w.s8x = reinterpret_cast<__half *>(w8 + 2 * split_bytes(K, B) + tscale_bytes(B));
    w.part = reinterpret_cast<float *>(w8 + 2 * split_bytes(K, B) + tscale_bytes(B) + s8x_bytes(K, B));
    return w;
}

cudaError_t launch_gemm_tc_split_done(const void *W, int N, int K, int B, float *y, void *ws, bool allow_split,
                                      cudaStream_t st)
{
    const TcWorkspace w = tc_workspace(ws, K, B);
    if (B <= kSmallMaxB) return launch_gemm_chunk(W, N, K, B, w.hi, w.lo, w.s8x, w.tscale, y, w.part, allow_split, st);
    const int splits = gemm_splits(B, N, K, allow_split);
    return launch_gemm_pair(W, N, K, B, w.hi, w.lo, w.s8x, w.tscale, splits > 1 ? w.part : y, y, splits, st);
}

cudaError_t launch_gemm_tc(const void *W, int N, int K, zq_q8_1 a, int B, float *y, void *ws, bool allow_split,
                           cudaStream_t st)
{
    const TcWorkspace w = tc_workspace(ws, K, B);
    cudaError_t e = launch_q8_split(a, K, B, w.hi, w.lo, w.tscale, w.s8x, st);
    if (e != cudaSuccess) return e;
    return launch_gemm_tc_split_done(W, N, K, B, y, ws, allow_split, st);
}

}  // namespace zq
