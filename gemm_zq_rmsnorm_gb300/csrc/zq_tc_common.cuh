// zq_tc_common.cuh -- pieces shared by the two tcgen05 kernels (the batched
// projection and the integer sub-block export): Q4_K nibble -> fp16
// conversion, bounded mbarrier waits that stop every role once one has failed,
// and the host-side tensor-map and activation-code helpers.
#pragma once

#include <cuda.h>

#include "zq_internal.cuh"
#include "zq_tc.cuh"

namespace zq {

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }

// Four fp16 values scale*q (two half2) from the four nibbles at bytes 0..3 of
// w, low (HIGH = false) or high nibble, in natural order.  The nibble is placed
// in the mantissa of 1024 (low) or 1024 + 16 q (high), so with scale = s,
// off = -1024 s (low) or scale = s/16, off = -64 s (high) one fused fp16
// operation gives s*q; exact while s*q fits in 11 bits.
template <bool HIGH>
__device__ __forceinline__ void nib4_to_h2(uint32_t w, __half2 scale, __half2 off, uint32_t &o0, uint32_t &o1)
{
    const uint32_t p0 = __byte_perm(w, 0, 0x4140);  // [b0, 0, b1, 0]
    const uint32_t p1 = __byte_perm(w, 0, 0x4342);  // [b2, 0, b3, 0]
    const uint32_t m = HIGH ? 0x00F000F0u : 0x000F000Fu;
    const uint32_t h0 = (p0 & m) | 0x64006400u;
    const uint32_t h1 = (p1 & m) | 0x64006400u;
    o0 = h2_bits(__hfma2(*reinterpret_cast<const __half2 *>(&h0), scale, off));
    o1 = h2_bits(__hfma2(*reinterpret_cast<const __half2 *>(&h1), scale, off));
}

// Bounded wait that also gives up at once when another role already failed.
// It sleeps between polls (woken by the phase's completion), so waiting
// warps leave the issue slots to the converters and the issuer.
static __device__ __noinline__ bool wait_ok(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                            unsigned int *status)
{
    if (*abort_flag) return false;
    const uint64_t t0 = global_ns();
    do {
        if (mbar_try_wait_sleep(bar, parity, kSleepNs)) return true;
        if (*abort_flag) return false;
    } while (global_ns() - t0 < kWaitLimitNs);
    flag_timeout(status);
    *abort_flag = 1;
    return false;
}

// One probe inline; the bounded loop only when the phase is not complete yet.
__device__ __forceinline__ bool wait_fast(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                          unsigned int *status)
{
    return mbar_try_wait(bar, parity) || wait_ok(bar, parity, abort_flag, status);
}

// One lane polls, then every lane acquires the completed phase itself.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                         unsigned int *status)
{
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = wait_fast(bar, parity, abort_flag, status);
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    if (ok) ok = wait_fast(bar, parity, abort_flag, status);
    return __all_sync(0xffffffffu, ok);
}

// 2-D tensor [rows][cols] of `esize`-byte elements, row stride cols * esize
// bytes, box box_cols x box_rows; elements outside the tensor read as zero.
cudaError_t make_tmap_2d(CUtensorMap *m, CUtensorMapDataType dt, uint32_t esize, const void *base, uint64_t cols,
                         uint64_t rows, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle sw);

// q8 activation codes -> fp16 (exact), n codes, n a multiple of 16.
cudaError_t launch_q8_to_f16(const int8_t *qs, __half *out, size_t n, cudaStream_t st);

// ---- shared by the projection kernels (q4k_gemm_tc.cu) -------------------
// Workspace: hi [B][K] binary16 | lo [B][K] binary16 | token scales [B] fp32
// | (B >= 17) the scaled, duplicated block sums s8x [B][K/16] binary16 |
// split-K partial sums [splits][split_stride(B, N)] fp32; regions padded to
// 256 bytes.
size_t split_bytes(int K, int B);
size_t tscale_bytes(int B);
// Floats between consecutive splits' partial sums: B * N rounded up to a
// multiple of 4, so that every split starts on a 16-byte boundary.
inline size_t split_stride(int B, int N) { return ((size_t)B * N + 3) & ~(size_t)3; }
// x' = q8 * d8 of every token split into exact binary16 hi + lo, with a
// per-token power-of-two scale that keeps the codes in binary16 range; with
// s8x non-null also each super-block's eight s8 values, scaled the same way,
// written twice ([B][K/16]).
cudaError_t launch_q8_split(zq_q8_1 a, int K, int B, __half *hi, __half *lo, float *tscale, __half *s8x,
                            cudaStream_t st);
// y[i] = sum over splits of part[s * split_stride + i] (in split order), i < n.
cudaError_t launch_splitk_reduce(const float *part, int splits, size_t n, float *y, cudaStream_t st);
// split-K count for the pair kernel (256 weight rows x 256 tokens per pair)
int choose_splits_pair(int B, int N, int K, int sms);

// the workspace's regions (layout above)
struct TcWorkspace {
    __half *hi, *lo, *s8x;
    float *tscale, *part;
};
TcWorkspace tc_workspace(void *ws, int K, int B);
// the projection on activations already split into the workspace
cudaError_t launch_gemm_tc_split_done(const void *W, int N, int K, int B, float *y, void *ws, bool allow_split,
                                      cudaStream_t st);
// largest B of the chunk kernel (q4k_gemm_chunk.cu); larger B run the pair kernel
constexpr int kSmallMaxB = 16;
// ---- CTA-pair projection (q4k_gemm_2sm.cu), B > kSmallMaxB ----------------
// out = y (splits == 1) or the partial-sum area; y receives the result.
cudaError_t launch_gemm_pair(const void *W, int N, int K, int B, const __half *hi, const __half *lo,
                             const __half *s8x, const float *tscale, float *out, float *y, int splits,
                             cudaStream_t st);
// ---- chunk projection (q4k_gemm_chunk.cu), 2 <= B <= kSmallMaxB ----------
// part: chunk_part_bytes(N, K, B) bytes of partial sums (allow_split), else
// unused: one CTA pair per 256-row tile and no partial sums.
size_t chunk_part_bytes(int N, int K, int B);
cudaError_t launch_gemm_chunk(const void *W, int N, int K, int B, const __half *hi, const __half *lo,
                              const __half *s8x, const float *tscale, float *y, float *part, bool allow_split,
                              cudaStream_t st);

}  // namespace zq
