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
// Rows of up to 576 blocks (K <= 18432): a persistent kernel, one block per
// thread, the token rows and gamma staged in shared memory by TMA (the next
// token's row loading during the current one) and, with the batched
// projection's activation split, the binary16 rows stored back by TMA
// (rmsnorm_q8_1_staged_kernel).  Wider rows of many tokens: one CTA per token
// with the row staged by TMA, one thread per block for the sums of squares
// and eight lanes per block for the rest, so every global access is
// coalesced (rmsnorm_q8_1_rows_kernel).  Otherwise one CTA per token with one
// thread per 32-element block (up to 1024 threads): every block's fma chain
// runs in parallel, the partials go through shared memory in block order, the
// block stays in registers between the two passes, and only the 256-slot
// sums and the tree are serial; rows of up to 2048 blocks (K <= 65536) give a
// thread two blocks, wider rows use a 256-thread kernel in which thread t
// owns the blocks of slot t.
//
// HBM roofline: reads B*K*4 bytes of x (+ K*4 of gamma, cached), writes
// B*K*(1 + 4/32) bytes.  At B = 1 the kernel is latency-bound.
#include <cuda.h>
#include <string.h>

#include "zq_async.cuh"
#include "zq_internal.cuh"
#include "zq_q8_1_pack.cuh"
#include "zq_tc.cuh"
#include "zq_tc_common.cuh"

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
// or all set): x' = q8 * d8 as exact binary16 hi + lo parts with the token's
// power-of-two scale 2^-k (tscale = 2^k, k from split_scale_exp, so that
// 127 * max d8 * 2^-k stays within binary16 range), and each super-block's
// eight s8 values scaled alike, twice.
struct SplitOut {
    __half *hi, *lo;
    float *tscale;
    __half *s8x;
};

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

// RMSNorm + Q8_1 (+ the activation split of the batched projection) with
// the token's row staged in shared memory: one CTA of 256 threads per token.
//  - One thread issues TMA copies of the row, 32 blocks (4 KB) each, as rows
//    of 128 bytes with the 128-byte swizzle (16-byte piece v of block b at
//    piece v ^ (b & 7)), each on its own mbarrier.
//  - Pass 1, one block per thread: thread t owns the blocks of slot t (t,
//    t + 256, ...) and reads each block's 32 values in order from shared
//    memory (the swizzle spreads a warp's reads over all banks); its running
//    sum is the slot sum itself.
//  - Pass 2, eight lanes per block (four values each), so that the reads of
//    gamma and every store are coalesced: (a) normalise in place and find
//    each block's amax and d8, and the token's largest d8; (b) after the
//    token's scale is known, quantise, sum the codes over the eight lanes,
//    and write the codes and, with the split, the binary16 hi/lo parts, the
//    token scale and s8x.
// Every value equals the thread-per-block kernels' (amax, the code sum and
// the element-wise steps do not depend on the order).
constexpr int kRowChunk = 32;      // blocks per TMA copy
constexpr int kRowsMinTokens = 5;  // codes-only calls with wider rows and at least this many tokens use it

__global__ void __launch_bounds__(256)
rmsnorm_q8_1_rows_kernel(const __grid_constant__ CUtensorMap tmap_x, const float *__restrict__ gamma, int K,
                         float eps, int8_t *__restrict__ qs, __half *__restrict__ dq, __half *__restrict__ sq,
                         SplitOut so, unsigned int *status)
{
    extern __shared__ uint8_t smem_raw[];
    float *xs = reinterpret_cast<float *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    __shared__ uint64_t bar[kMaxThreads / kRowChunk];
    __shared__ float slot_s[256];
    __shared__ float red_s[8];
    __shared__ float r_s;
    __shared__ int fail_s;
    const int t = threadIdx.x;
    const int nblk = K >> 5, nchunk = (nblk + kRowChunk - 1) / kRowChunk;
    float *d_s = xs + (size_t)nchunk * kRowChunk * 32;   // d8 of each block, fp32
    const size_t tok = blockIdx.x;
    if (t == 0) {
        for (int c = 0; c < nchunk; ++c) mbar_init(&bar[c], 1);
        fail_s = 0;
        fence_mbar_init();
    }
    __syncthreads();
    pdl_wait();   // x may come from the previous kernel; the outputs may still be read by it
    pdl_launch_dependents();
    if (t == 0) {
        prefetch_tmap(&tmap_x);
        for (int c = 0; c < nchunk; ++c) {
            mbar_arrive_expect_tx(&bar[c], kRowChunk * 128);
            tma_load_2d(xs + (size_t)c * kRowChunk * 32, &tmap_x, 0, (int)(tok * nblk) + kRowChunk * c, &bar[c]);
        }
    }

    // pass 1: the slot sum of p_b
    float slot = 0.0f;
    bool ok = true;
    for (int b = t; b < nblk; b += 256) {
        if (!(ok = mbar_wait(&bar[b / kRowChunk], 0, status))) break;
        const float4 *row = reinterpret_cast<const float4 *>(xs + 32 * b);
        float part = 0.0f;
#pragma unroll
        for (int v = 0; v < 8; ++v) {
            const float4 f = row[v ^ (b & 7)];
            part = __fmaf_rn(f.x, f.x, part);
            part = __fmaf_rn(f.y, f.y, part);
            part = __fmaf_rn(f.z, f.z, part);
            part = __fmaf_rn(f.w, f.w, part);
        }
        slot = __fadd_rn(slot, part);
    }
    if (!ok) fail_s = 1;
    slot_s[t] = slot;
    __syncthreads();
    if (fail_s) {
        // a copy did not land in time (status raised): let copies still in
        // flight finish before the CTA's shared memory goes away
        for (int c = 0; c < nchunk; ++c) mbar_wait_for(&bar[c], 0, nullptr, 1000000ull);
        return;
    }
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

    // pass 2a: lanes 8g .. 8g + 7 of warp w take block 4w + g (+ 32 j),
    // piece `sub` of it; the warp's four blocks are 512 contiguous bytes
    // (nblk is a multiple of 8, so a warp's blocks are all in range or none)
    const int warp = t >> 5, lane = t & 31, sub = lane & 7;
    const int b0 = 4 * warp + (lane >> 3);
    // gamma of the lane's next four blocks stays in flight (an L2 round trip
    // per block would otherwise set the pace)
    float4 gq[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
        gq[u] = b0 + 32 * u < nblk ? __ldg(reinterpret_cast<const float4 *>(gamma + 32 * (b0 + 32 * u)) + sub)
                                   : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    float m = 0.0f;
    for (int j = 0; b0 + 32 * j < nblk; j += 4) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int b = b0 + 32 * (j + u);
            if (b >= nblk) break;
            const float4 g = gq[u];
            if (b + 128 < nblk) gq[u] = __ldg(reinterpret_cast<const float4 *>(gamma + 32 * (b + 128)) + sub);
            float4 *cell = reinterpret_cast<float4 *>(xs + 32 * b) + (sub ^ (b & 7));
            float4 f = *cell;
            f.x = __fmul_rn(__fmul_rn(f.x, r), g.x);
            f.y = __fmul_rn(__fmul_rn(f.y, r), g.y);
            f.z = __fmul_rn(__fmul_rn(f.z, r), g.z);
            f.w = __fmul_rn(__fmul_rn(f.w, r), g.w);
            *cell = f;
            float a = fmaxf(fmaxf(fabsf(f.x), fabsf(f.y)), fmaxf(fabsf(f.z), fabsf(f.w)));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
            const float d = __fdiv_rn(a, 127.0f);
            if (sub == 0) d_s[b] = d;
            m = fmaxf(m, __half2float(__float2half_rn(d)));
        }
    }
    // the token's power-of-two scale 2^-k from its largest d8
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if (lane == 0) red_s[warp] = m;
    __syncthreads();
    m = red_s[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) m = fmaxf(m, red_s[w]);
    const int k = split_scale_exp(m);
    const float down = pow2_exact(-k);
    if (so.hi != nullptr && t == 0) so.tscale[tok] = pow2_exact(k);

    // pass 2b: the codes of the lane's four values, the block's code sum, s8
#pragma unroll 2
    for (int b = b0; b < nblk; b += 32) {
        const float4 f = reinterpret_cast<const float4 *>(xs + 32 * b)[sub ^ (b & 7)];
        const float d = d_s[b];
        const float id = (d != 0.0f) ? __fdiv_rn(1.0f, d) : 0.0f;
        const float xv[4] = {f.x, f.y, f.z, f.w};
        int q[4];
        uint32_t word = 0;
        int sum = 0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const float qf = fminf(fmaxf(roundf(__fmul_rn(xv[c], id)), -127.0f), 127.0f);
            q[c] = (int)qf;
            sum += q[c];
            word |= ((uint32_t)(q[c] & 0xFF)) << (8 * c);
        }
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        sum += __shfl_xor_sync(0xffffffffu, sum, 4);
        const __half dh = __float2half_rn(d);
        const __half sh = __float2half_rn(__fmul_rn(d, (float)sum));
        const size_t e0 = tok * K + 32 * (size_t)b + 4 * sub;   // the lane's first element
        if (qs != nullptr) {
            *reinterpret_cast<uint32_t *>(qs + e0) = word;
            if (sub == 0) {
                dq[tok * nblk + b] = dh;
                sq[tok * nblk + b] = sh;
            }
        }
        if (so.hi != nullptr) {
            // x' = q8 * d8 * 2^-k (exact in fp32) as binary16 hi + lo
            const float dv = __fmul_rn(__half2float(dh), down);
            const float a0 = __fmul_rn((float)q[0], dv), a1 = __fmul_rn((float)q[1], dv);
            const float a2 = __fmul_rn((float)q[2], dv), a3 = __fmul_rn((float)q[3], dv);
            const __half2 h01 = __floats2half2_rn(a0, a1), h23 = __floats2half2_rn(a2, a3);
            const float2 b01 = __half22float2(h01), b23 = __half22float2(h23);
            const __half2 l01 = __floats2half2_rn(__fsub_rn(a0, b01.x), __fsub_rn(a1, b01.y));
            const __half2 l23 = __floats2half2_rn(__fsub_rn(a2, b23.x), __fsub_rn(a3, b23.y));
            *reinterpret_cast<uint2 *>(so.hi + e0) = make_uint2(h2_bits(h01), h2_bits(h23));
            *reinterpret_cast<uint2 *>(so.lo + e0) = make_uint2(h2_bits(l01), h2_bits(l23));
            if (sub == 0) {
                const __half sv = __float2half_rn(__fmul_rn(__half2float(sh), down));
                __half *sx = so.s8x + tok * (K / 16) + 16 * (b >> 3) + (b & 7);
                sx[0] = sv;
                sx[8] = sv;
            }
        }
    }
}

// Persistent RMSNorm + Q8_1 (+ the activation split) for rows of up to
// kStagedMaxBlocks blocks (K <= 18432), one block per thread throughout:
//  - a TMA warp copies γ once and the tokens' rows into two row buffers
//    (4 KB per copy, 128-byte rows, 128-byte swizzle), the next token's row
//    loading while the CTA works on the current one; with the split it also
//    stores the token's binary16 hi and lo rows from shared memory (64-byte
//    rows, 64-byte swizzle: 16-byte piece q of block b at q ^ ((b >> 1) & 3));
//  - compute thread t owns block t: its fma chain, then the slot sums and
//    the tree in the canonical order, then normalisation and packing from
//    shared memory (the swizzles keep a warp's 128-byte rows on distinct
//    banks), codes and s8x to global memory, hi/lo into the row buffer it
//    has finished reading.
// All global traffic of the row is whole TMA boxes; the thread-per-block
// arithmetic is the same as rmsnorm_q8_1_kernel's, so the bytes are too.
constexpr int kStagedMaxBlocks = 576;
constexpr int kStagedMaxChunks = kStagedMaxBlocks / kRowChunk;

struct StagedMaps {
    CUtensorMap x, g;            // x [B * nblk][32] fp32, γ [nblk][32] fp32; boxes of 32 rows
    CUtensorMap hi32, lo32;      // hi, lo [B * nblk][32] binary16; boxes of 32 rows
    CUtensorMap hi8, lo8;        // the same, boxes of 8 rows (a row's last blocks)
};

__global__ void __launch_bounds__(kStagedMaxBlocks + 32)
rmsnorm_q8_1_staged_kernel(const __grid_constant__ StagedMaps maps, int B, int K, float eps,
                           int8_t *__restrict__ qs, __half *__restrict__ dq, __half *__restrict__ sq, SplitOut so,
                           unsigned int *status)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    __shared__ uint64_t gbar[kStagedMaxChunks], xbar[2][kStagedMaxChunks], sfree[2];
    __shared__ float part_s[kStagedMaxBlocks];
    __shared__ float slot_s[256];
    __shared__ float red_s[kStagedMaxBlocks / 32];
    __shared__ float r_s;
    __shared__ int fail_s;

    const int t = threadIdx.x;
    const int nblk = K >> 5, nchunk = (nblk + kRowChunk - 1) / kRowChunk;
    const int nc = (int)blockDim.x - 32, ncw = nc >> 5;   // compute threads; the last warp moves data
    const size_t buf_bytes = (size_t)nchunk * kRowChunk * 128;
    uint8_t *const gs = sm;
    uint8_t *const xb0 = sm + buf_bytes;
    const bool split = so.hi != nullptr;
    const int G = (int)gridDim.x;

    if (t == 0) {
        for (int c = 0; c < nchunk; ++c) {
            mbar_init(&gbar[c], 1);
            mbar_init(&xbar[0][c], 1);
            mbar_init(&xbar[1][c], 1);
        }
        mbar_init(&sfree[0], (uint32_t)ncw);   // buffer s read (and, with the split, staged) by every compute warp
        mbar_init(&sfree[1], (uint32_t)ncw);
        fail_s = 0;
        fence_mbar_init();
    }
    __syncthreads();
    pdl_wait();   // x may come from the previous kernel; the outputs may still be read by it
    pdl_launch_dependents();

    if (t >= nc) {
        // ---------------------------------------------------- TMA warp
        if (t == nc) {
            prefetch_tmap(&maps.x);
            prefetch_tmap(&maps.g);
            for (int c = 0; c < nchunk; ++c) {
                mbar_arrive_expect_tx(&gbar[c], kRowChunk * 128);
                tma_load_2d(gs + (size_t)c * kRowChunk * 128, &maps.g, 0, kRowChunk * c, &gbar[c]);
            }
            auto load_x = [&](int j) {
                const int tok = (int)blockIdx.x + j * G, s = j & 1;
                uint8_t *xb = xb0 + (size_t)s * buf_bytes;
                for (int c = 0; c < nchunk; ++c) {
                    mbar_arrive_expect_tx(&xbar[s][c], kRowChunk * 128);
                    tma_load_2d(xb + (size_t)c * kRowChunk * 128, &maps.x, 0, tok * nblk + kRowChunk * c,
                                &xbar[s][c]);
                }
            };
            load_x(0);
            if ((int)blockIdx.x + G < B) load_x(1);
            for (int j = 0;; ++j) {
                const int tok = (int)blockIdx.x + j * G, s = j & 1;
                if (tok >= B) break;
                if (!wait_fast(&sfree[s], (uint32_t)(j >> 1) & 1u, &fail_s, status)) break;
                if (split) {
                    const uint8_t *hs = xb0 + (size_t)s * buf_bytes, *ls = hs + buf_bytes / 2;
                    const int full = nblk / kRowChunk;
                    for (int c = 0; c < full; ++c) {
                        tma_store_2d(&maps.hi32, 0, tok * nblk + kRowChunk * c, hs + (size_t)c * kRowChunk * 64);
                        tma_store_2d(&maps.lo32, 0, tok * nblk + kRowChunk * c, ls + (size_t)c * kRowChunk * 64);
                    }
                    for (int r0 = kRowChunk * full; r0 < nblk; r0 += 8) {
                        tma_store_2d(&maps.hi8, 0, tok * nblk + r0, hs + (size_t)r0 * 64);
                        tma_store_2d(&maps.lo8, 0, tok * nblk + r0, ls + (size_t)r0 * 64);
                    }
                    bulk_commit();
                    bulk_wait_read<0>();   // the buffer may take the next row
                }
                if (tok + 2 * G < B) load_x(j + 2);
            }
            bulk_wait<0>();
        }
    } else {
        // ---------------------------------------------------- compute threads
        const int warp = t >> 5, lane = t & 31;
        const bool own = t < nblk;
        for (int j = 0;; ++j) {
            const int tok = (int)blockIdx.x + j * G, s = j & 1;
            if (tok >= B) break;
            uint8_t *const xb = xb0 + (size_t)s * buf_bytes;
            bool ok = true;
            float xr[32];
            if (own) {
                ok = wait_fast(&xbar[s][t >> 5], (uint32_t)(j >> 1) & 1u, &fail_s, status);
                if (ok && j == 0) ok = wait_fast(&gbar[t >> 5], 0, &fail_s, status);
                if (ok) {
                    const float4 *row = reinterpret_cast<const float4 *>(xb + (size_t)128 * t);
#pragma unroll
                    for (int v = 0; v < 8; ++v) {
                        const float4 f = row[v ^ (t & 7)];
                        xr[4 * v + 0] = f.x;
                        xr[4 * v + 1] = f.y;
                        xr[4 * v + 2] = f.z;
                        xr[4 * v + 3] = f.w;
                    }
                    float part = 0.0f;
#pragma unroll
                    for (int i = 0; i < 32; ++i) part = __fmaf_rn(xr[i], xr[i], part);
                    part_s[t] = part;
                }
            }
            // one decision for every compute thread: a copy that did not land
            // in time ends the CTA's work (the status word is raised)
            if (named_bar_or(1, (uint32_t)nc, !ok)) {
                fail_s = 1;
                break;
            }
            if (t < 256) {
                float slot = 0.0f;
                for (int b = t; b < nblk; b += 256) slot = __fadd_rn(slot, part_s[b]);
                slot_s[t] = slot;
            }
            named_bar(1, (uint32_t)nc);
#pragma unroll
            for (int off = 128; off >= 32; off >>= 1) {
                if (t < off) slot_s[t] = __fadd_rn(slot_s[t], slot_s[t + off]);
                named_bar(1, (uint32_t)nc);
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
            named_bar(1, (uint32_t)nc);
            const float r = r_s;
            Q8Block pk{};
            if (own) {
                const float4 *grow = reinterpret_cast<const float4 *>(gs + (size_t)128 * t);
#pragma unroll
                for (int v = 0; v < 8; ++v) {
                    const float4 w = grow[v ^ (t & 7)];
                    xr[4 * v + 0] = __fmul_rn(__fmul_rn(xr[4 * v + 0], r), w.x);
                    xr[4 * v + 1] = __fmul_rn(__fmul_rn(xr[4 * v + 1], r), w.y);
                    xr[4 * v + 2] = __fmul_rn(__fmul_rn(xr[4 * v + 2], r), w.z);
                    xr[4 * v + 3] = __fmul_rn(__fmul_rn(xr[4 * v + 3], r), w.w);
                }
                pk = q8_1_pack(xr);
                if (qs != nullptr) {
                    const size_t o = (size_t)tok * nblk + t;
                    uint4 *dst = reinterpret_cast<uint4 *>(qs + (size_t)tok * K + 32 * t);
                    dst[0] = pk.q0;
                    dst[1] = pk.q1;
                    dq[o] = pk.d;
                    sq[o] = pk.s;
                }
            }
            if (split) {
                // the token's power-of-two scale 2^-k from its largest d8
                float m = own ? fabsf(__half2float(pk.d)) : 0.0f;
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
                if (lane == 0) red_s[warp] = m;
                named_bar(1, (uint32_t)nc);   // (also: every compute thread has read its x from the buffer)
                m = red_s[0];
                for (int w = 1; w < ncw; ++w) m = fmaxf(m, red_s[w]);
                const int k = split_scale_exp(m);
                const float down = pow2_exact(-k);
                if (t == 0) so.tscale[tok] = pow2_exact(k);
                if (own) {
                    // x' = q8 * d8 * 2^-k (exact in fp32) as binary16 hi + lo,
                    // into the buffer's hi and lo halves (64-byte swizzle)
                    const float dv = __fmul_rn(__half2float(pk.d), down);
                    const uint32_t w[8] = {pk.q0.x, pk.q0.y, pk.q0.z, pk.q0.w, pk.q1.x, pk.q1.y, pk.q1.z, pk.q1.w};
                    uint8_t *hrow = xb + (size_t)64 * t, *lrow = hrow + buf_bytes / 2;
                    const int sw = (t >> 1) & 3;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {   // values 8q .. 8q + 7
                        uint32_t oh[4], ol[4];
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj) {
                            const uint32_t x2 = w[2 * q + (jj >> 1)] >> (16 * (jj & 1));
                            const float a0 = __fmul_rn((float)(int8_t)(x2 & 0xFFu), dv);
                            const float a1 = __fmul_rn((float)(int8_t)((x2 >> 8) & 0xFFu), dv);
                            const __half2 vh = __floats2half2_rn(a0, a1);
                            const float2 back = __half22float2(vh);
                            oh[jj] = h2_bits(vh);
                            ol[jj] = h2_bits(__floats2half2_rn(__fsub_rn(a0, back.x), __fsub_rn(a1, back.y)));
                        }
                        *reinterpret_cast<uint4 *>(hrow + 16 * (q ^ sw)) = make_uint4(oh[0], oh[1], oh[2], oh[3]);
                        *reinterpret_cast<uint4 *>(lrow + 16 * (q ^ sw)) = make_uint4(ol[0], ol[1], ol[2], ol[3]);
                    }
                    const __half sv = __float2half_rn(__fmul_rn(__half2float(pk.s), down));
                    __half *sx = so.s8x + (size_t)tok * (K / 16) + 16 * (t >> 3) + (t & 7);
                    sx[0] = sv;
                    sx[8] = sv;
                    fence_async_smem();   // the TMA store reads the staging through the async proxy
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sfree[s]);
        }
    }
    if (*reinterpret_cast<volatile int *>(&fail_s)) {
        // a role gave up: let copies already issued land before the CTA's
        // shared memory goes away
        const uint64_t tw = global_ns();
        while (global_ns() - tw < 200000ull) {
        }
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

static size_t rows_smem_bytes(int K)
{
    const int nblk = K / 32, nchunk = (nblk + kRowChunk - 1) / kRowChunk;
    return 1024 + (size_t)nchunk * kRowChunk * 128 + (size_t)nblk * 4;
}

static size_t staged_smem_bytes(int K)
{
    const int nblk = K / 32, nchunk = (nblk + kRowChunk - 1) / kRowChunk;
    return 1024 + 3 * (size_t)nchunk * kRowChunk * 128;   // γ and two row buffers
}

static cudaError_t launch_staged(const float *x, const float *gamma, int B, int K, float eps, int8_t *qs,
                                 __half *dq, __half *sq, SplitOut so, cudaStream_t st)
{
    const int nblk = K / 32;
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(gamma)) & 15u) return cudaErrorInvalidValue;
    StagedMaps maps;
    memset(&maps, 0, sizeof(maps));
    const uint64_t rows = (uint64_t)B * nblk;
    cudaError_t e;
    if ((e = make_tmap_2d(&maps.x, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, x, 32, rows, 32, kRowChunk,
                          CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess ||
        (e = make_tmap_2d(&maps.g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, gamma, 32, (uint64_t)nblk, 32, kRowChunk,
                          CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
        return e;
    if (so.hi != nullptr) {
        const CUtensorMapDataType f16 = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
        if ((e = make_tmap_2d(&maps.hi32, f16, 2, so.hi, 32, rows, 32, kRowChunk, CU_TENSOR_MAP_SWIZZLE_64B)) !=
                cudaSuccess ||
            (e = make_tmap_2d(&maps.lo32, f16, 2, so.lo, 32, rows, 32, kRowChunk, CU_TENSOR_MAP_SWIZZLE_64B)) !=
                cudaSuccess ||
            (e = make_tmap_2d(&maps.hi8, f16, 2, so.hi, 32, rows, 32, 8, CU_TENSOR_MAP_SWIZZLE_64B)) != cudaSuccess ||
            (e = make_tmap_2d(&maps.lo8, f16, 2, so.lo, 32, rows, 32, 8, CU_TENSOR_MAP_SWIZZLE_64B)) != cudaSuccess)
            return e;
    }
    const int threads = (nblk > 256 ? (nblk + 31) / 32 * 32 : 256) + 32;
    const size_t smem = staged_smem_bytes(K);
    static bool attr = false;
    if (!attr) {
        if ((e = cudaFuncSetAttribute(rmsnorm_q8_1_staged_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)staged_smem_bytes(32 * kStagedMaxBlocks))) != cudaSuccess)
            return e;
        attr = true;
    }
    // CTAs per SM for this row width, found once per width
    static int occ_of[kStagedMaxBlocks / 8 + 1];
    int &occ = occ_of[nblk / 8];
    if (occ == 0) {
        if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, rmsnorm_q8_1_staged_kernel, threads, smem)) !=
            cudaSuccess)
            return e;
        if (occ < 1) return cudaErrorInvalidConfiguration;
    }
    const long long cap = (long long)num_sms() * occ;
    const int grid = (int)(B < cap ? B : cap);
    return launch_pdl(rmsnorm_q8_1_staged_kernel, dim3(grid), dim3(threads), smem, st, maps, B, K, eps, qs, dq, sq, so,
                      device_status_word());
}

cudaError_t launch_rmsnorm_q8_1(const float *x, const float *gamma, int B, int K, float eps, zq_q8_1 out,
                                cudaStream_t st)
{
    const int nblk = K / 32;
    __half *dq = reinterpret_cast<__half *>(out.d);
    __half *sq = reinterpret_cast<__half *>(out.s);
    // rows of up to kStagedMaxBlocks blocks: the persistent staged kernel;
    // wider rows of many tokens: the row-staged kernel (coalesced global
    // accesses); otherwise one thread per block, no staging
    if (nblk <= kStagedMaxBlocks)
        return launch_staged(x, gamma, B, K, eps, out.qs, dq, sq, SplitOut{nullptr, nullptr, nullptr, nullptr}, st);
    // (the row-staged kernel's eight-lane groups need K % 256 == 0: a warp's
    // four blocks are then all in the row or all past it)
    if (B >= kRowsMinTokens && nblk <= kMaxThreads && nblk % 8 == 0)
        return launch_rmsnorm_q8_1_split(x, gamma, B, K, eps, &out, nullptr, nullptr, nullptr, nullptr, st);
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
    if (nblk > kMaxThreads) return cudaErrorInvalidValue;   // K > 32768
    // the split's 8-row stores, and the row-staged kernel's eight-lane
    // groups, need whole groups of eight blocks (K % 256 == 0)
    if ((hi != nullptr || nblk > kStagedMaxBlocks) && nblk % 8 != 0) return cudaErrorInvalidValue;
    if (nblk <= kStagedMaxBlocks)
        return launch_staged(x, gamma, B, K, eps, out ? out->qs : nullptr,
                             out ? reinterpret_cast<__half *>(out->d) : nullptr,
                             out ? reinterpret_cast<__half *>(out->s) : nullptr, SplitOut{hi, lo, tscale, s8x}, st);
    if (reinterpret_cast<uintptr_t>(x) & 15u) return cudaErrorInvalidValue;
    CUtensorMap tx;
    cudaError_t e = make_tmap_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, x, 32, (uint64_t)B * nblk, 32, kRowChunk,
                                 CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
    const size_t smem = rows_smem_bytes(K);
    static size_t attr = 0;
    if (smem > attr) {
        if ((e = cudaFuncSetAttribute(rmsnorm_q8_1_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)rows_smem_bytes(32768))) != cudaSuccess)
            return e;
        attr = rows_smem_bytes(32768);
    }
    int8_t *qs = out ? out->qs : nullptr;
    __half *dq = out ? reinterpret_cast<__half *>(out->d) : nullptr;
    __half *sq = out ? reinterpret_cast<__half *>(out->s) : nullptr;
    return launch_pdl(rmsnorm_q8_1_rows_kernel, dim3(B), dim3(256), smem, st, tx, gamma, K, eps, qs, dq, sq,
                      SplitOut{hi, lo, tscale, s8x}, device_status_word());
}

}  // namespace zq
