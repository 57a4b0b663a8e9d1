// q4k_gemm_tc.cu -- batched Q4_K x Q8_1 projection on the tcgen05 tensor
// cores (B >= 2 tokens).
//
// MIInfer README, "Current phase": token-batched chunk projections for
// prefill, a raw int8 GEMM as the speed bound of the native Q4_K path, and
// tensor-core prefill; ZINC docs "ROCm backend", "Build and verify": matrix-
// core prefill tiles that consume the Q4 weights directly.
//
// The contraction is exact in integers per 32-weight sub-block, as the
// projection's definition requires:
//   y[t][n] = sum_b d_b[n] * ( sum_j d8[t][bj] * sc_j[n] * I[t][n][bj] )
//           - sum_b dmin_b[n] * ( sum_j m_j[n] * s8[t][bj] ).
// sm_103a has no int8 tcgen05 MMA, so both operands are fed as fp16 holding
// small integers exactly: A = activation codes q8 (|q8| <= 127), B = sc_j*q4
// (<= 945, exact in binary16).  Every product and every partial sum of a
// sub-block is an integer below 2^22, so the fp32 tensor-core accumulator
// holds sc_j * I exactly.  Per sub-block the MMA (M = 128 tokens, N = 128
// weight rows, K = 32 as two K = 16 steps) writes one of two TMEM buffers;
// epilogue warps read it back and accumulate inner += d8 * D in registers
// (d8 is a per-lane scalar: TMEM lanes are tokens).  Once per super-block a
// second MMA forms sum_j s8[t][bj] * m_j[n] (K = 16: eight mins and eight
// zeros) in TMEM, and the epilogue folds acc += d_b*inner - dmin_b*minsum into
// an fp32 accumulator kept in TMEM.
//
// Warp roles (14 warps): 0 TMA producer (fp16 activation tiles, s8 tiles),
// 1 MMA issuer + TMEM owner, 2-5 weight converters (Q4_K bytes -> sc*q fp16
// in the 128-byte-swizzled K-major layout, mins, d/dmin), 6-13 epilogue
// (2 column groups of 64 x 4 lane quarters).  Every wait is bounded.
#include <cuda.h>

#include "zq_internal.cuh"
#include "zq_tc.cuh"

namespace zq {
namespace {

constexpr int BM = 128;               // tokens per tile (TMEM lanes)
constexpr int BN = 128;               // weight rows per tile (TMEM columns)
constexpr int kStages = 3;            // half super-block (K = 128) stages
constexpr int kAtomBytes = 128 * 128; // 128 rows x 64 fp16 (128 B), 128-byte swizzle
constexpr int kStageBytes = 4 * kAtomBytes;  // A: 2 atoms, B: 2 atoms
constexpr int kMinBytes = 128 * 32;   // 128 rows x 16 fp16, 32-byte swizzle
constexpr int kWarps = 14;
constexpr int kThreads = kWarps * 32;
constexpr int kConvWarp0 = 2, kConvWarps = 4;
constexpr int kEpiWarp0 = 6, kEpiWarps = 8;
constexpr int kEpiCols = BN / (kEpiWarps / 4);   // 64 columns per epilogue thread
constexpr uint32_t kIdesc = idesc_f16_f32(BM, BN);
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColD0 = 0, kColD1 = 128, kColMin = 256, kColAcc = 384;

struct Smem {
    // offsets from the 1024-aligned base
    static constexpr size_t stage(int s) { return (size_t)s * kStageBytes; }
    static constexpr size_t a_atom(int s, int a) { return stage(s) + (size_t)a * kAtomBytes; }
    static constexpr size_t b_atom(int s, int a) { return stage(s) + (size_t)(2 + a) * kAtomBytes; }
    static constexpr size_t amin(int i) { return (size_t)kStages * kStageBytes + (size_t)i * 2 * kMinBytes; }
    static constexpr size_t bmin(int i) { return amin(i) + kMinBytes; }
    static constexpr size_t dd(int i) { return amin(2) + (size_t)i * BN * 8; }
    static constexpr size_t bars() { return dd(2); }
    static constexpr int kNumBars = 3 * kStages + 7 * 2 + 2;  // stage x3, seven pairs, two singles
    static constexpr size_t tmem_slot() { return bars() + kNumBars * 8; }
    static constexpr size_t total() { return tmem_slot() + 16 + 1024; }  // + alignment slack
};

struct Bars {
    uint64_t *a_full, *b_full, *st_empty;      // [kStages]
    uint64_t *amin_full, *bmin_full, *min_empty;  // [2]
    uint64_t *mma_done, *epi_done;             // [2]
    uint64_t *dd_full, *dd_free;               // [2]
    uint64_t *min_done, *min_free;
};

struct GemmParams {
    const uint8_t *W;
    int N, K, B, nb;
    uint32_t rowbytes;
    int t_tiles;
    const __half *d8;   // Q8_1 scales [B][K/32]
    float *y;           // [B][N]
    int32_t *isums;     // debug export [B][N][K/32] (or null)
    unsigned int *status;
};

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }

// Four fp16 sc*q values (two half2) from four nibbles at bytes 0..3 of w,
// low (HIGH = false) or high nibble, in natural order.  (1024 + q) * sc - 1024 * sc
// and (1024 + 16 q) * sc/16 - 64 * sc are exact in one fused rounding.
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

// bounded wait that also gives up at once when another role already failed
__device__ __forceinline__ bool wait_ok(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                        unsigned int *status)
{
    if (*abort_flag) return false;
    for (uint32_t i = 0; i < kSpinLimit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 1023u) == 1023u && *abort_flag) return false;
    }
    flag_timeout(status);
    *abort_flag = 1;
    return false;
}

// one lane polls, then every lane acquires the completed phase itself
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                         unsigned int *status)
{
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = wait_ok(bar, parity, abort_flag, status);
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    if (ok) ok = wait_ok(bar, parity, abort_flag, status);
    return __all_sync(0xffffffffu, ok);
}

template <bool DEBUG>
__global__ void __maxnreg__(128)
q4k_gemm_wide_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_s,
                     const GemmParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    __shared__ volatile int abort_s;

    uint64_t *barmem = reinterpret_cast<uint64_t *>(sm + Smem::bars());
    Bars bar;
    bar.a_full = barmem;
    bar.b_full = barmem + kStages;
    bar.st_empty = barmem + 2 * kStages;
    bar.amin_full = barmem + 3 * kStages;
    bar.bmin_full = bar.amin_full + 2;
    bar.min_empty = bar.amin_full + 4;
    bar.mma_done = bar.amin_full + 6;
    bar.epi_done = bar.mma_done + 2;
    bar.dd_full = bar.mma_done + 4;
    bar.dd_free = bar.mma_done + 6;
    bar.min_done = bar.mma_done + 8;
    bar.min_free = bar.mma_done + 9;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + Smem::tmem_slot());

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int t_tile = blockIdx.x % p.t_tiles;
    const int n_tile = blockIdx.x / p.t_tiles;
    const int t0 = t_tile * BM;
    const int n0 = n_tile * BN;
    const int nb = p.nb;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bar.a_full[s], 1);
            mbar_init(&bar.b_full[s], kConvWarps);
            mbar_init(&bar.st_empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar.amin_full[i], 1);
            mbar_init(&bar.bmin_full[i], kConvWarps);
            mbar_init(&bar.min_empty[i], 1);
            mbar_init(&bar.mma_done[i], 1);
            mbar_init(&bar.epi_done[i], kEpiWarps);
            mbar_init(&bar.dd_full[i], kConvWarps);
            mbar_init(&bar.dd_free[i], kEpiWarps);
        }
        mbar_init(bar.min_done, 1);
        mbar_init(bar.min_free, kEpiWarps);
        abort_s = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------------------------------------------- TMA producer
        if (lane == 0) {
            prefetch_tmap(&tmap_a);
            prefetch_tmap(&tmap_s);
            for (int q = 0; q < 2 * nb; ++q) {
                const int b = q >> 1, h = q & 1;
                const int slot = q % kStages, round = q / kStages;
                if (round > 0 && !wait_ok(&bar.st_empty[slot], (round & 1) ^ 1, &abort_s, p.status)) break;
                mbar_arrive_expect_tx(&bar.a_full[slot], 2 * kAtomBytes);
                const int k0 = 256 * b + 128 * h;
                tma_load_2d(sm + Smem::a_atom(slot, 0), &tmap_a, k0, t0, &bar.a_full[slot]);
                tma_load_2d(sm + Smem::a_atom(slot, 1), &tmap_a, k0 + 64, t0, &bar.a_full[slot]);
                if (h == 0) {
                    const int mi = b & 1, use = b >> 1;
                    if (use > 0 && !wait_ok(&bar.min_empty[mi], (use & 1) ^ 1, &abort_s, p.status)) break;
                    mbar_arrive_expect_tx(&bar.amin_full[mi], kMinBytes);
                    tma_load_2d(sm + Smem::amin(mi), &tmap_s, 8 * b, t0, &bar.amin_full[mi]);
                }
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t base = smem_u32(sm);
            for (int q = 0; q < 2 * nb; ++q) {
                const int b = q >> 1, h = q & 1;
                const int slot = q % kStages, round = q / kStages;
                if (!wait_ok(&bar.a_full[slot], round & 1, &abort_s, p.status)) break;
                if (!wait_ok(&bar.b_full[slot], round & 1, &abort_s, p.status)) break;
                tc_fence_after();
                bool fail = false;
                for (int jj = 0; jj < 4; ++jj) {
                    const int s = 8 * b + 4 * h + jj;
                    const int buf = s & 1, use = s >> 1;
                    if (use > 0 && !wait_ok(&bar.epi_done[buf], (use - 1) & 1, &abort_s, p.status)) {
                        fail = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_at = base + (uint32_t)Smem::a_atom(slot, jj >> 1);
                    const uint32_t b_at = base + (uint32_t)Smem::b_atom(slot, jj >> 1);
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk) {
                        const uint32_t off = (uint32_t)((jj & 1) * 64 + kk * 32);
                        mma_f16(tmem + (buf ? kColD1 : kColD0), smem_desc(a_at + off, 16, 1024, kLayoutSw128),
                                smem_desc(b_at + off, 16, 1024, kLayoutSw128), kIdesc, (uint32_t)kk);
                    }
                    mma_commit(&bar.mma_done[buf]);
                }
                if (fail) break;
                mma_commit(&bar.st_empty[slot]);
                if (h == 1) {
                    const int mi = b & 1, use = b >> 1;
                    if (!wait_ok(&bar.amin_full[mi], use & 1, &abort_s, p.status)) break;
                    if (!wait_ok(&bar.bmin_full[mi], use & 1, &abort_s, p.status)) break;
                    if (b > 0 && !wait_ok(bar.min_free, (b - 1) & 1, &abort_s, p.status)) break;
                    tc_fence_after();
                    mma_f16(tmem + kColMin,
                            smem_desc(base + (uint32_t)Smem::amin(mi), 16, 256, kLayoutSw32),
                            smem_desc(base + (uint32_t)Smem::bmin(mi), 16, 256, kLayoutSw32), kIdesc, 0u);
                    mma_commit(bar.min_done);
                    mma_commit(&bar.min_empty[mi]);
                }
            }
        }
    } else if (warp < kEpiWarp0) {
        // ---------------------------------------------------- converters
        const int r = (warp - kConvWarp0) * 32 + lane;   // row within the tile
        const int row = n0 + r;
        const bool valid = row < p.N;
        const uint8_t *rowp = p.W + (size_t)(valid ? row : 0) * p.rowbytes;
        for (int q = 0; q < 2 * nb; ++q) {
            const int b = q >> 1, h = q & 1;
            const int slot = q % kStages, round = q / kStages;
            if (round > 0 && !warp_wait(&bar.st_empty[slot], (round & 1) ^ 1, &abort_s, p.status)) break;
            const uint8_t *blk = rowp + (size_t)b * kQ4KBlockBytes;
            uint4 hdr = make_uint4(0, 0, 0, 0), nib[4];
            if (valid) {
                hdr = ld_stream_u4(blk);
#pragma unroll
                for (int i = 0; i < 4; ++i) nib[i] = ld_stream_u4(blk + 16 + 64 * h + 16 * i);
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i) nib[i] = make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int a = 0; a < 2; ++a) {
                const int jl = 4 * h + 2 * a;   // sub-blocks jl (low nibbles), jl + 1 (high)
                uint32_t sc0, sc1, mdummy;
                q4k_scale_min(hdr.y, hdr.z, hdr.w, jl, sc0, mdummy);
                q4k_scale_min(hdr.y, hdr.z, hdr.w, jl + 1, sc1, mdummy);
                const float scl = DEBUG ? 1.0f : (float)sc0;
                const float sch = DEBUG ? 1.0f : (float)sc1;
                const __half2 s_lo = __float2half2_rn(scl), o_lo = __float2half2_rn(-1024.0f * scl);
                const __half2 s_hi = __float2half2_rn(sch * 0.0625f), o_hi = __float2half2_rn(-64.0f * sch);
                const uint32_t wv[8] = {nib[2 * a].x,     nib[2 * a].y,     nib[2 * a].z,     nib[2 * a].w,
                                        nib[2 * a + 1].x, nib[2 * a + 1].y, nib[2 * a + 1].z, nib[2 * a + 1].w};
                uint8_t *atom = sm + Smem::b_atom(slot, a) + (size_t)r * 128;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint4 lo, hi;
                    nib4_to_h2<false>(wv[2 * c], s_lo, o_lo, lo.x, lo.y);
                    nib4_to_h2<false>(wv[2 * c + 1], s_lo, o_lo, lo.z, lo.w);
                    nib4_to_h2<true>(wv[2 * c], s_hi, o_hi, hi.x, hi.y);
                    nib4_to_h2<true>(wv[2 * c + 1], s_hi, o_hi, hi.z, hi.w);
                    *reinterpret_cast<uint4 *>(atom + ((c ^ (r & 7)) << 4)) = lo;
                    *reinterpret_cast<uint4 *>(atom + (((c + 4) ^ (r & 7)) << 4)) = hi;
                }
            }
            if (h == 0) {
                const int mi = b & 1, use = b >> 1;
                // mins as the B operand of the per-super-block min MMA
                if (use > 0 && !warp_wait(&bar.min_empty[mi], (use & 1) ^ 1, &abort_s, p.status)) break;
                uint32_t mn[8], scd;
#pragma unroll
                for (int j = 0; j < 8; ++j) q4k_scale_min(hdr.y, hdr.z, hdr.w, j, scd, mn[j]);
                uint4 m0;
                m0.x = h2_bits(__floats2half2_rn((float)mn[0], (float)mn[1]));
                m0.y = h2_bits(__floats2half2_rn((float)mn[2], (float)mn[3]));
                m0.z = h2_bits(__floats2half2_rn((float)mn[4], (float)mn[5]));
                m0.w = h2_bits(__floats2half2_rn((float)mn[6], (float)mn[7]));
                uint8_t *bm = sm + Smem::bmin(mi) + (size_t)r * 32;
                const int sw = (r >> 2) & 1;
                *reinterpret_cast<uint4 *>(bm + ((0 ^ sw) << 4)) = m0;
                *reinterpret_cast<uint4 *>(bm + ((1 ^ sw) << 4)) = make_uint4(0, 0, 0, 0);
                // d, dmin for the epilogue
                if (use > 0 && !warp_wait(&bar.dd_free[mi], (use - 1) & 1, &abort_s, p.status)) break;
                const float2 dd = valid ? __half22float2(*reinterpret_cast<const __half2 *>(&hdr.x))
                                        : make_float2(0.0f, 0.0f);
                reinterpret_cast<float2 *>(sm + Smem::dd(mi))[r] = dd;
                fence_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&bar.bmin_full[mi]);
                    mbar_arrive(&bar.dd_full[mi]);
                }
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar.b_full[slot]);
        }
    } else {
        // ---------------------------------------------------- epilogue
        const int e = warp - kEpiWarp0;
        const int cg = e >> 2;                    // column group: columns 64cg .. 64cg+63
        const int quarter = warp & 3;             // TMEM lanes 32*quarter .. +31
        const int tl = 32 * quarter + lane;       // token within the tile
        const int tok = t0 + tl;
        const bool tvalid = tok < p.B;
        const uint32_t lane_base = tmem + ((uint32_t)(32 * quarter) << 16);
        const int nsub = nb * 8;
        float inner[kEpiCols];
#pragma unroll
        for (int c = 0; c < kEpiCols; ++c) inner[c] = 0.0f;
        uint4 d8raw = make_uint4(0, 0, 0, 0);
        if (tvalid && !DEBUG) d8raw = __ldg(reinterpret_cast<const uint4 *>(p.d8 + (size_t)tok * nsub));
        bool ok = true;
        for (int b = 0; b < nb && ok; ++b) {
            uint4 d8next = make_uint4(0, 0, 0, 0);
            if (tvalid && !DEBUG && b + 1 < nb)
                d8next = __ldg(reinterpret_cast<const uint4 *>(p.d8 + (size_t)tok * nsub + 8 * (b + 1)));
            for (int j = 0; j < 8; ++j) {
                const int s = 8 * b + j;
                const int buf = s & 1, use = s >> 1;
                if (!warp_wait(&bar.mma_done[buf], use & 1, &abort_s, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t w2 = (j < 4) ? ((j < 2) ? d8raw.x : d8raw.y) : ((j < 6) ? d8raw.z : d8raw.w);
                const uint16_t hb = (j & 1) ? (uint16_t)(w2 >> 16) : (uint16_t)(w2 & 0xFFFFu);
                const float d8 = __half2float(__ushort_as_half(hb));
#pragma unroll
                for (int chunk = 0; chunk < kEpiCols / 32; ++chunk) {
                    uint32_t r[32];
                    tmem_ld32(lane_base + (buf ? kColD1 : kColD0) + kEpiCols * cg + 32 * chunk, r);
                    tmem_wait_ld();
                    if (DEBUG) {
                        if (tvalid) {
#pragma unroll
                            for (int c = 0; c < 32; ++c) {
                                const int n = n0 + kEpiCols * cg + 32 * chunk + c;
                                if (n < p.N)
                                    p.isums[((size_t)tok * p.N + n) * nsub + s] = (int32_t)__uint_as_float(r[c]);
                            }
                        }
                    } else {
#pragma unroll
                        for (int c = 0; c < 32; ++c)
                            inner[32 * chunk + c] = fmaf(d8, __uint_as_float(r[c]), inner[32 * chunk + c]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar.epi_done[buf]);
            }
            if (!ok) break;
            d8raw = d8next;
            // super-block end: acc = acc + d_b * inner - dmin_b * minsum
            const int mi = b & 1, use = b >> 1;
            if (!warp_wait(bar.min_done, b & 1, &abort_s, p.status)) break;
            if (!warp_wait(&bar.dd_full[mi], use & 1, &abort_s, p.status)) break;
            tc_fence_after();
            if (!DEBUG) {
                const float2 *dd = reinterpret_cast<const float2 *>(sm + Smem::dd(mi)) + kEpiCols * cg;
#pragma unroll
                for (int q16 = 0; q16 < kEpiCols / 16; ++q16) {
                    uint32_t mr[16], ar[16];
                    tmem_ld16(lane_base + kColMin + kEpiCols * cg + 16 * q16, mr);
                    if (b > 0) tmem_ld16(lane_base + kColAcc + kEpiCols * cg + 16 * q16, ar);
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const float2 v = dd[16 * q16 + c];
                        float acc = b > 0 ? __uint_as_float(ar[c]) : 0.0f;
                        acc = fmaf(v.x, inner[16 * q16 + c], acc);
                        acc = fmaf(-v.y, __uint_as_float(mr[c]), acc);
                        ar[c] = __float_as_uint(acc);
                    }
                    tmem_st16(lane_base + kColAcc + kEpiCols * cg + 16 * q16, ar);
                }
                tmem_wait_st();
#pragma unroll
                for (int c = 0; c < kEpiCols; ++c) inner[c] = 0.0f;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bar.min_free);
                mbar_arrive(&bar.dd_free[mi]);
            }
        }
        if (ok && !abort_s && !DEBUG) {
            uint32_t ar[16];
#pragma unroll
            for (int q16 = 0; q16 < kEpiCols / 16; ++q16) {
                tmem_ld16(lane_base + kColAcc + kEpiCols * cg + 16 * q16, ar);
                tmem_wait_ld();
                if (tvalid) {
                    float *yrow = p.y + (size_t)tok * p.N;
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const int n = n0 + kEpiCols * cg + 16 * q16 + c;
                        if (n < p.N) yrow[n] = __uint_as_float(ar[c]);
                    }
                }
            }
        }
    }
    __syncwarp();  // producer / issuer warps: reconverge with their lane 0
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
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

// ---------------------------------------------------------------- host side
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

// 2-D fp16 tensor [rows][cols] (row stride = cols*2 bytes), box box_cols x box_rows
cudaError_t make_tmap(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows, uint32_t box_cols,
                      uint32_t box_rows, CUtensorMapSwizzle sw)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

size_t g_attr_bytes[64][2];

template <bool DEBUG>
cudaError_t launch_wide(const void *W, int N, int K, zq_q8_1 a, int B, float *y, int32_t *isums, void *ws,
                        cudaStream_t st)
{
    __half *a16 = static_cast<__half *>(ws);
    const size_t n16 = (size_t)B * K / 16;
    q8_to_f16_kernel<<<(unsigned)((n16 + 255) / 256), 256, 0, st>>>(a.qs, a16, n16);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    CUtensorMap ta, ts;
    if ((e = make_tmap(&ta, a16, (uint64_t)K, (uint64_t)B, 64, BM, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
        return e;
    if ((e = make_tmap(&ts, a.s, (uint64_t)K / 32, (uint64_t)B, 16, BM, CU_TENSOR_MAP_SWIZZLE_32B)) != cudaSuccess)
        return e;
    GemmParams p{};
    p.W = static_cast<const uint8_t *>(W);
    p.N = N;
    p.K = K;
    p.B = B;
    p.nb = K / 256;
    p.rowbytes = (uint32_t)p.nb * kQ4KBlockBytes;
    p.t_tiles = (B + BM - 1) / BM;
    p.d8 = reinterpret_cast<const __half *>(a.d);
    p.y = y;
    p.isums = isums;
    p.status = device_status_word();
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    const size_t smem = Smem::total();
    if (g_attr_bytes[dev][DEBUG] < smem) {
        e = cudaFuncSetAttribute(q4k_gemm_wide_kernel<DEBUG>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        g_attr_bytes[dev][DEBUG] = smem;
    }
    const long long grid = (long long)p.t_tiles * ((N + BN - 1) / BN);
    q4k_gemm_wide_kernel<DEBUG><<<(unsigned)grid, kThreads, smem, st>>>(ta, ts, p);
    return cudaGetLastError();
}

}  // namespace

size_t gemm_tc_workspace_bytes(int N, int K, int B)
{
    (void)N;
    if (B <= 1) return 0;
    return (size_t)B * K * sizeof(__half);
}

cudaError_t launch_gemm_tc_wide(const void *W, int N, int K, zq_q8_1 a, int B, float *y, int32_t *isums, void *ws,
                                cudaStream_t st)
{
    if (isums) return launch_wide<true>(W, N, K, a, B, nullptr, isums, ws, st);
    return launch_wide<false>(W, N, K, a, B, y, nullptr, ws, st);
}

cudaError_t launch_gemm_tc_narrow(const void *W, int N, int K, zq_q8_1 a, int B, float *y, int32_t *isums,
                                  void *ws, cudaStream_t st)
{
    // chunk sizes run on the same tensor-core kernel: one 128-token tile whose
    // rows beyond B are zero-filled by the TMA and never stored
    return launch_gemm_tc_wide(W, N, K, a, B, y, isums, ws, st);
}

}  // namespace zq
