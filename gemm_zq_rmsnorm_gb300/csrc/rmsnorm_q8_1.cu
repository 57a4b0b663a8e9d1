// rmsnorm_q8_1.cu -- fused RMSNorm + Q8_1 activation packing.
//
// ZINC docs "ROCm backend", "Build and verify": RMS normalisation and Q8
// activation packing share one wide per-token kernel, saving a second read of
// the activations and a launch.
//
// The sum of squares follows the library's fixed order: per 32-element block
// a fused multiply-add chain over its squares in index order (p_b); 256 slots,
// slot t the sum of p_b over b = t (mod 256) in increasing b; a pairwise tree
// over the slots.  Every floating-point step is an explicitly rounded IEEE
// fp32 operation (__fmaf_rn, __fadd_rn, __fmul_rn, __fdiv_rn, __fsqrt_rn), so
// codes and scales are reproducible bit for bit.
//
// One CTA per token with one thread per 32-element block (up to 1024
// threads): every block's fma chain runs in parallel, the partials go through
// shared memory in block order, the block stays in registers between the two
// passes, and only the 256-slot sums and the tree are serial.  Rows of up to
// 2048 blocks (K <= 65536) give a thread two blocks; wider rows use a 256-thread
// kernel in which thread t owns the blocks of slot t.
//
// HBM roofline: reads B*K*4 bytes of x (+ K*4 of gamma, cached), writes
// B*K*(1 + 4/32) bytes.  At B = 1 the kernel is latency-bound.
#include "zq_async.cuh"
#include "zq_internal.cuh"
#include "zq_q8_1_pack.cuh"

namespace zq {
namespace {

constexpr int kMaxThreads = 1024;
constexpr int kMaxBlocks = 2048;   // K <= 65536 on this path

// Quantise one 32-value block (already normalised) to Q8_1 and store it.
__device__ __forceinline__ void pack_block(const float (&xh)[32], int8_t *qdst, __half *dq, __half *sq)
{
    const Q8Block o = q8_1_pack(xh);
    uint4 *dst = reinterpret_cast<uint4 *>(qdst);
    dst[0] = o.q0;
    dst[1] = o.q1;
    *dq = o.d;
    *sq = o.s;
}

// Optional outputs of the batched projection's activation split (all null,
// or all set; only when every block has a thread of its own): x' = q8 * d8
// as exact binary16 hi + lo parts with the token's power-of-two scale 2^-k
// (tscale = 2^k, k >= 0 the least that keeps 127 * max d8 within binary16
// range), and each super-block's eight s8 values scaled alike, twice.
struct SplitOut {
    __half *hi, *lo;
    float *tscale;
    __half *s8x;
};

// One block's share of the activation split, with the token's scale
// down = 2^-k applied: its 32 values x' = q8 * d8 * 2^-k as exact binary16
// hi + lo parts, and its scaled s8 value in both halves of its super-block's
// 16-entry s8x row (the same numbers as q8_split_kernel derives from the
// stored codes).
__device__ __forceinline__ void split_block(const Q8Block &pk, int b, float down, int K, SplitOut so)
{
    const float dv = __half2float(pk.d) * down;
    const uint32_t w[8] = {pk.q0.x, pk.q0.y, pk.q0.z, pk.q0.w, pk.q1.x, pk.q1.y, pk.q1.z, pk.q1.w};
    uint4 *dh = reinterpret_cast<uint4 *>(so.hi + (size_t)blockIdx.x * K + 32 * b);
    uint4 *dl = reinterpret_cast<uint4 *>(so.lo + (size_t)blockIdx.x * K + 32 * b);
#pragma unroll
    for (int q = 0; q < 4; ++q) {   // codes 8q .. 8q + 7
        uint32_t oh[4], ol[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {   // codes 8q + 2j, 8q + 2j + 1
            const uint32_t x2 = w[2 * q + (j >> 1)] >> (16 * (j & 1));
            const float a0 = (float)(int8_t)(x2 & 0xFFu) * dv, a1 = (float)(int8_t)((x2 >> 8) & 0xFFu) * dv;
            const __half2 vh = __floats2half2_rn(a0, a1);
            const float2 back = __half22float2(vh);
            oh[j] = *reinterpret_cast<const uint32_t *>(&vh);
            const __half2 vl = __floats2half2_rn(a0 - back.x, a1 - back.y);
            ol[j] = *reinterpret_cast<const uint32_t *>(&vl);
        }
        dh[q] = make_uint4(oh[0], oh[1], oh[2], oh[3]);
        dl[q] = make_uint4(ol[0], ol[1], ol[2], ol[3]);
    }
    const __half sv = __float2half_rn(__half2float(pk.s) * down);
    __half *sx = so.s8x + (size_t)blockIdx.x * (K / 16) + 16 * (b >> 3) + (b & 7);
    sx[0] = sv;
    sx[8] = sv;
}

__global__ void __launch_bounds__(kMaxThreads)
rmsnorm_q8_1_kernel(const float *__restrict__ x, const float *__restrict__ gamma, int K, float eps,
                    int8_t *__restrict__ qs, __half *__restrict__ dq, __half *__restrict__ sq)
{
    __shared__ float part_s[kMaxBlocks];   // p_b, in block order
    __shared__ float slot_s[256];
    __shared__ float r_s;

    const int t = threadIdx.x;
    const int nthr = blockDim.x;
    const int nblk = K >> 5;
    const float *xt = x + (size_t)blockIdx.x * K;
    const bool one = nblk <= nthr;   // one block per thread: keep it in registers
    pdl_wait();                  // x may come from the previous kernel; Q8_1 may still be read by it
    pdl_launch_dependents();

    // pass 1: p_b for every block
    float xr[32];
    for (int b = t; b < nblk; b += nthr) {
        const float4 *p = reinterpret_cast<const float4 *>(xt + 32 * b);
#pragma unroll
        for (int v = 0; v < 8; ++v) {
            const float4 f = __ldg(p + v);
            xr[4 * v + 0] = f.x;
            xr[4 * v + 1] = f.y;
            xr[4 * v + 2] = f.z;
            xr[4 * v + 3] = f.w;
        }
        float part = 0.0f;
#pragma unroll
        for (int i = 0; i < 32; ++i) part = __fmaf_rn(xr[i], xr[i], part);
        part_s[b] = part;
    }
    __syncthreads();
    // slot t: blocks t, t + 256, ... added in increasing b, from +0
    if (t < 256) {
        float slot = 0.0f;
        for (int b = t; b < nblk; b += 256) slot = __fadd_rn(slot, part_s[b]);
        slot_s[t] = slot;
    }
    __syncthreads();
    // pairwise tree, off = 128 .. 32 through shared memory, 16 .. 1 in a warp
#pragma unroll
    for (int off = 128; off >= 32; off >>= 1) {
        if (t < off) slot_s[t] = __fadd_rn(slot_s[t], slot_s[t + off]);
        __syncthreads();
    }
    if (t < 32) {
        float v = slot_s[t];
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) v = __fadd_rn(v, __shfl_down_sync(0xffffffffu, v, off));
        if (t == 0) {
            const float mean = __fdiv_rn(v, (float)K);
            r_s = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, eps)));
        }
    }
    __syncthreads();
    const float r = r_s;

    // pass 2: normalise and pack each block
    for (int b = t; b < nblk; b += nthr) {
        if (!one) {
            const float4 *p = reinterpret_cast<const float4 *>(xt + 32 * b);
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                const float4 f = __ldg(p + v);
                xr[4 * v + 0] = f.x;
                xr[4 * v + 1] = f.y;
                xr[4 * v + 2] = f.z;
                xr[4 * v + 3] = f.w;
            }
        }
        const float4 *g = reinterpret_cast<const float4 *>(gamma + 32 * b);
#pragma unroll
        for (int v = 0; v < 8; ++v) {   // normalise in place
            const float4 w = __ldg(g + v);
            xr[4 * v + 0] = __fmul_rn(__fmul_rn(xr[4 * v + 0], r), w.x);
            xr[4 * v + 1] = __fmul_rn(__fmul_rn(xr[4 * v + 1], r), w.y);
            xr[4 * v + 2] = __fmul_rn(__fmul_rn(xr[4 * v + 2], r), w.z);
            xr[4 * v + 3] = __fmul_rn(__fmul_rn(xr[4 * v + 3], r), w.w);
        }
        const size_t o = (size_t)blockIdx.x * nblk + b;
        pack_block(xr, qs + (size_t)blockIdx.x * K + 32 * b, dq + o, sq + o);
    }
}

// Rows wider than kMaxBlocks blocks: one CTA of 256 threads per token, thread
// t owning the blocks t, t+256, ... (its slot), re-reading x in pass 2.
__global__ void __launch_bounds__(256)
rmsnorm_q8_1_wide_kernel(const float *__restrict__ x, const float *__restrict__ gamma, int K, float eps,
                         int8_t *__restrict__ qs, __half *__restrict__ dq, __half *__restrict__ sq)
{
    __shared__ float slot_s[256];
    __shared__ float r_s;
    const int t = threadIdx.x;
    const int nblk = K >> 5;
    const float *xt = x + (size_t)blockIdx.x * K;
    pdl_wait();
    pdl_launch_dependents();
    float slot = 0.0f;
    for (int b = t; b < nblk; b += 256) {
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
#pragma unroll
    for (int off = 128; off >= 32; off >>= 1) {
        if (t < off) slot_s[t] = __fadd_rn(slot_s[t], slot_s[t + off]);
        __syncthreads();
    }
    if (t < 32) {
        float v = slot_s[t];
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) v = __fadd_rn(v, __shfl_down_sync(0xffffffffu, v, off));
        if (t == 0) {
            const float mean = __fdiv_rn(v, (float)K);
            r_s = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, eps)));
        }
    }
    __syncthreads();
    const float r = r_s;
    for (int b = t; b < nblk; b += 256) {
        const float4 *p = reinterpret_cast<const float4 *>(xt + 32 * b);
        const float4 *g = reinterpret_cast<const float4 *>(gamma + 32 * b);
        float xh[32];
#pragma unroll
        for (int v = 0; v < 8; ++v) {
            const float4 f = __ldg(p + v);
            const float4 w = __ldg(g + v);
            xh[4 * v + 0] = __fmul_rn(__fmul_rn(f.x, r), w.x);
            xh[4 * v + 1] = __fmul_rn(__fmul_rn(f.y, r), w.y);
            xh[4 * v + 2] = __fmul_rn(__fmul_rn(f.z, r), w.z);
            xh[4 * v + 3] = __fmul_rn(__fmul_rn(f.w, r), w.w);
        }
        const size_t o = (size_t)blockIdx.x * nblk + b;
        pack_block(xh, qs + (size_t)blockIdx.x * K + 32 * b, dq + o, sq + o);
    }
}

// RMSNorm + Q8_1 + the activation split for the batched projection, rows
// of up to 256 * MB blocks.  One CTA of 256 threads per token, thread t
// owning the blocks of slot t (t, t + 256, ...), so its running sum of their
// p_b in increasing b is the slot sum itself; at most 64 registers a thread,
// so four tokens' CTAs share an SM and 512 tokens run in one wave.  A single
// block stays in registers between the passes; with more, all of them are
// prefetched into L2 while the first loads and read again in pass 2.  The
// packed codes wait in shared memory until the token's largest d8 is known.
template <int MB>
__global__ void __launch_bounds__(256, 4)
rmsnorm_q8_1_split_kernel(const float *__restrict__ x, const float *__restrict__ gamma, int K, float eps,
                          int8_t *__restrict__ qs, __half *__restrict__ dq, __half *__restrict__ sq, SplitOut so)
{
    __shared__ float slot_s[256];
    __shared__ float r_s;
    __shared__ float dmax_s[8];
    __shared__ uint4 kq_s[MB][2][256];   // codes of block t + 256 i
    __shared__ __half2 kds_s[MB][256];   // its (d, s)
    const int t = threadIdx.x;
    const int nblk = K >> 5;
    const int mine = t < nblk ? (nblk - 1 - t) / 256 + 1 : 0;
    const float *xt = x + (size_t)blockIdx.x * K;
    pdl_wait();   // x may come from the previous kernel; the outputs may still be read by it
    pdl_launch_dependents();
#pragma unroll
    for (int i = 0; i < MB; ++i)
        if (i < mine) {
            if (i > 0) asm volatile("prefetch.global.L2 [%0];" ::"l"(xt + 32 * (t + 256 * i)));
            asm volatile("prefetch.global.L1 [%0];" ::"l"(gamma + 32 * (t + 256 * i)));
        }

    // pass 1: the slot sum of p_b
    float xr[32];
    float slot = 0.0f;
#pragma unroll
    for (int i = 0; i < MB; ++i) {
        if (i >= mine) break;
        const float4 *p = reinterpret_cast<const float4 *>(xt + 32 * (t + 256 * i));
        float part = 0.0f;
        if (MB == 1) {
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                const float4 f = __ldg(p + v);
                xr[4 * v + 0] = f.x;
                xr[4 * v + 1] = f.y;
                xr[4 * v + 2] = f.z;
                xr[4 * v + 3] = f.w;
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) part = __fmaf_rn(xr[j], xr[j], part);
        } else {
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                const float4 f = __ldg(p + v);
                part = __fmaf_rn(f.x, f.x, part);
                part = __fmaf_rn(f.y, f.y, part);
                part = __fmaf_rn(f.z, f.z, part);
                part = __fmaf_rn(f.w, f.w, part);
            }
        }
        slot = __fadd_rn(slot, part);
    }
    slot_s[t] = slot;
    __syncthreads();
#pragma unroll
    for (int off = 128; off >= 32; off >>= 1) {
        if (t < off) slot_s[t] = __fadd_rn(slot_s[t], slot_s[t + off]);
        __syncthreads();
    }
    if (t < 32) {
        float v = slot_s[t];
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) v = __fadd_rn(v, __shfl_down_sync(0xffffffffu, v, off));
        if (t == 0) {
            const float mean = __fdiv_rn(v, (float)K);
            r_s = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, eps)));
        }
    }
    __syncthreads();
    const float r = r_s;

    // pass 2: normalise and pack, tracking the largest |d8|
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < MB; ++i) {
        if (i >= mine) break;
        const int b = t + 256 * i;
        if (MB > 1) {
            const float4 *p = reinterpret_cast<const float4 *>(xt + 32 * b);
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                const float4 f = __ldg(p + v);
                xr[4 * v + 0] = f.x;
                xr[4 * v + 1] = f.y;
                xr[4 * v + 2] = f.z;
                xr[4 * v + 3] = f.w;
            }
        }
        const float4 *g = reinterpret_cast<const float4 *>(gamma + 32 * b);
#pragma unroll
        for (int v = 0; v < 8; ++v) {
            const float4 w = __ldg(g + v);
            xr[4 * v + 0] = __fmul_rn(__fmul_rn(xr[4 * v + 0], r), w.x);
            xr[4 * v + 1] = __fmul_rn(__fmul_rn(xr[4 * v + 1], r), w.y);
            xr[4 * v + 2] = __fmul_rn(__fmul_rn(xr[4 * v + 2], r), w.z);
            xr[4 * v + 3] = __fmul_rn(__fmul_rn(xr[4 * v + 3], r), w.w);
        }
        const Q8Block pk = q8_1_pack(xr);
        m = fmaxf(m, fabsf(__half2float(pk.d)));
        if (qs != nullptr) {
            const size_t o = (size_t)blockIdx.x * nblk + b;
            uint4 *dst = reinterpret_cast<uint4 *>(qs + (size_t)blockIdx.x * K + 32 * b);
            dst[0] = pk.q0;
            dst[1] = pk.q1;
            dq[o] = pk.d;
            sq[o] = pk.s;
        }
        kq_s[i][0][t] = pk.q0;
        kq_s[i][1][t] = pk.q1;
        kds_s[i][t] = __halves2half2(pk.d, pk.s);
    }

    // the token's power-of-two scale 2^-k from its largest d8
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if ((t & 31) == 0) dmax_s[t >> 5] = m;
    __syncthreads();
    m = dmax_s[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) m = fmaxf(m, dmax_s[w]);
    const int k = split_scale_exp(m);   // 127 * m bounds every |x'| of the token
    const float down = pow2_exact(-k);
    if (t == 0) so.tscale[blockIdx.x] = pow2_exact(k);
#pragma unroll
    for (int i = 0; i < MB; ++i) {
        if (i >= mine) break;
        Q8Block pk;
        pk.q0 = kq_s[i][0][t];
        pk.q1 = kq_s[i][1][t];
        const __half2 ds = kds_s[i][t];
        pk.d = __low2half(ds);
        pk.s = __high2half(ds);
        split_block(pk, t + 256 * i, down, K, so);
    }
}
// h = silu(g) * u packed to Q8_1: one thread per 32-value block
__global__ void __launch_bounds__(256)
silu_mul_q8_1_kernel(const float *__restrict__ g, const float *__restrict__ u, int K, int8_t *__restrict__ qs,
                     __half *__restrict__ dq, __half *__restrict__ sq)
{
    pdl_wait();   // g and u may come from the previous kernel; the codes may still be read by it
    pdl_launch_dependents();
    const int nblk = K >> 5;
    const int b = blockIdx.y * blockDim.x + threadIdx.x;
    if (b >= nblk) return;
    const size_t off = (size_t)blockIdx.x * K + 32 * (size_t)b;
    const float4 *pg = reinterpret_cast<const float4 *>(g + off);
    const float4 *pu = reinterpret_cast<const float4 *>(u + off);
    float h[32];
#pragma unroll
    for (int v = 0; v < 8; ++v) {
        const float4 a = __ldg(pg + v), c = __ldg(pu + v);
        h[4 * v + 0] = silu_mul(a.x, c.x);
        h[4 * v + 1] = silu_mul(a.y, c.y);
        h[4 * v + 2] = silu_mul(a.z, c.z);
        h[4 * v + 3] = silu_mul(a.w, c.w);
    }
    const size_t o = (size_t)blockIdx.x * nblk + b;
    pack_block(h, qs + off, dq + o, sq + o);
}

}  // namespace

cudaError_t launch_silu_mul_q8_1(const float *g, const float *u, int B, int K, zq_q8_1 out, cudaStream_t st)
{
    const int nblk = K / 32;
    const dim3 grid((unsigned)B, (unsigned)((nblk + 255) / 256));
    return launch_pdl(silu_mul_q8_1_kernel, grid, dim3(256), 0, st, g, u, K, out.qs,
                      reinterpret_cast<__half *>(out.d), reinterpret_cast<__half *>(out.s));
}

cudaError_t launch_rmsnorm_q8_1(const float *x, const float *gamma, int B, int K, float eps, zq_q8_1 out,
                                cudaStream_t st)
{
    const int nblk = K / 32;
    __half *dq = reinterpret_cast<__half *>(out.d);
    __half *sq = reinterpret_cast<__half *>(out.s);
    if (nblk <= kMaxBlocks) {
        int threads = nblk < kMaxThreads ? (nblk + 31) / 32 * 32 : kMaxThreads;
        if (threads < 256) threads = 256;   // the slot tree needs 256 threads
        return launch_pdl(rmsnorm_q8_1_kernel, dim3(B), dim3(threads), 0, st, x, gamma, K, eps, out.qs, dq, sq);
    }
    return launch_pdl(rmsnorm_q8_1_wide_kernel, dim3(B), dim3(256), 0, st, x, gamma, K, eps, out.qs, dq, sq);
}

cudaError_t launch_rmsnorm_q8_1_split(const float *x, const float *gamma, int B, int K, float eps,
                                      const zq_q8_1 *out, __half *hi, __half *lo, float *tscale, __half *s8x,
                                      cudaStream_t st)
{
    const int nblk = K / 32;
    int8_t *qs = out ? out->qs : nullptr;
    __half *dq = out ? reinterpret_cast<__half *>(out->d) : nullptr;
    __half *sq = out ? reinterpret_cast<__half *>(out->s) : nullptr;
    const SplitOut so{hi, lo, tscale, s8x};
    switch ((nblk + 255) / 256) {
    case 1: return launch_pdl(rmsnorm_q8_1_split_kernel<1>, dim3(B), dim3(256), 0, st, x, gamma, K, eps, qs, dq, sq, so);
    case 2: return launch_pdl(rmsnorm_q8_1_split_kernel<2>, dim3(B), dim3(256), 0, st, x, gamma, K, eps, qs, dq, sq, so);
    case 3: return launch_pdl(rmsnorm_q8_1_split_kernel<3>, dim3(B), dim3(256), 0, st, x, gamma, K, eps, qs, dq, sq, so);
    case 4: return launch_pdl(rmsnorm_q8_1_split_kernel<4>, dim3(B), dim3(256), 0, st, x, gamma, K, eps, qs, dq, sq, so);
    default: return cudaErrorInvalidValue;   // K > 32768
    }
}

}  // namespace zq
