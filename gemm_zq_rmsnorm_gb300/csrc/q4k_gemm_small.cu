// q4k_gemm_small.cu -- Q4_K x Q8_1 projection of a few tokens (2 <= B <= 16)
// on the tcgen05 tensor cores.
//
// MIInfer README, "Current phase": token-batched chunk projections (chunks of
// four tokens) that read each weight once for the whole chunk.
//
// A chunk is bound by HBM: the weights are read once and every weight serves
// only B <= 16 tokens.  The batched kernel's 128-token tiles would waste the
// tensor cores and, worse, pay one tile's full pipeline per 64 values of K.
// Here the roles are swapped: the MMA's M side is 128 weight rows (A,
// converted to binary16 sc*q4 by converter warps) and its N side the B tokens
// padded to 16, twice: the binary16 hi and lo halves of q8*d8 (as in the
// batched kernel) sit in columns 0-15 and 16-31 of one N = 32 operand, so
// one 128 x 32 x 16 MMA covers both halves and a stage holds half a
// super-block of weights.  Every product is exact; X (one super-block, hi
// and lo columns) and the min product Mn land in a 4-super-block TMEM ring,
// and one epilogue thread per weight row folds
// acc[t] += d_b * (Xhi[t] + Xlo[t]) - dmin_b * 2^-k_t * Mn[t] in registers.
//
// Warp roles (14 warps): 0 TMA producer (hi/lo activation tiles, s8 tiles,
// raw Q4_K tiles three super-blocks ahead), 1 MMA issuer + TMEM owner, 2-9
// converters (half a weight row each: Q4_K nibbles -> sc*q binary16 in the
// 128-byte-swizzled K-major layout; mins and d/-dmin once per super-block),
// 10-13 epilogue (one TMEM lane quarter each).  Every wait is bounded.
//
// Measured (5120 -> 17408, B = 16): ~1.1 TB/s.  Each 128 x 32 x 16 MMA holds
// the issuing thread for ~90 cycles whatever N, and the eight converter warps
// take ~1000-2000 cycles per stage, so a stage of 16K weights costs ~1500
// cycles instead of the ~440 at which the weights would stream at full HBM
// bandwidth.
#include <cuda.h>

#include "zq_internal.cuh"
#include "zq_tc.cuh"
#include "zq_tc_common.cuh"

namespace zq {
namespace {

constexpr int SR = 128;                  // weight rows per tile (TMEM lanes, MMA M)
constexpr int ST = 16;                   // token columns (MMA N)
constexpr int kStages = 3;               // operand stages of K = 128 (four sub-blocks)
constexpr int kWAtom = SR * 128;         // 128 rows x 64 binary16 (128 B), 128-byte swizzle: 16 KB
constexpr int kWStageBytes = 2 * kWAtom; // K = 128
constexpr int kAAtom = ST * 128;         // 16 tokens x 64 binary16: 2 KB
constexpr int kAStageBytes = 4 * kAAtom; // per 64-wide K chunk c: hi atom, then lo atom (32 rows)
constexpr int kRawSlots = 4;             // raw Q4_K tiles in flight (super-blocks)
constexpr int kRawBytes = SR * kQ4KBlockBytes;
constexpr int kWMinBytes = SR * 32;      // 128 rows x 16 binary16, 32-byte swizzle
constexpr int kAMinBytes = ST * 32;      // 16 tokens x 16 binary16, 32-byte swizzle
constexpr int kRing = 4;                 // super-blocks in TMEM: X (32 columns) and Mn (16), 64 per slot
constexpr int kSlotCols = 64;
constexpr int kWarps = 14;
constexpr int kThreads = kWarps * 32;
constexpr int kConvWarp0 = 2, kConvWarps = 8;
constexpr int kEpiWarp0 = 10, kEpiWarps = 4;
constexpr uint32_t kIdesc = idesc_f16_f32(SR, 2 * ST);      // hi and lo token columns
constexpr uint32_t kIdescMin = idesc_f16_f32(SR, ST);
constexpr uint32_t kTmemCols = 256;
static_assert(kConvWarps * 32 == 2 * SR, "two converter threads per weight row");
static_assert(kRing * kSlotCols <= (int)kTmemCols && 3 * ST <= kSlotCols, "ring fits the allocation");

struct Smem {
    static constexpr size_t w_stage(int s) { return (size_t)s * kWStageBytes; }
    static constexpr size_t a_stage(int s) { return w_stage(kStages) + (size_t)s * kAStageBytes; }
    static constexpr size_t raw(int i) { return a_stage(kStages) + (size_t)i * kRawBytes; }
    static constexpr size_t wmin(int i) { return raw(kRawSlots) + (size_t)i * kWMinBytes; }
    static constexpr size_t amin(int i) { return wmin(2) + (size_t)i * kAMinBytes; }
    static constexpr size_t dd(int i) { return amin(2) + (size_t)i * SR * 8; }   // d[SR], then -dmin[SR]
    static constexpr size_t bars() { return dd(2); }
    static constexpr int kNumBars = 2 * kStages + 2 * kRawSlots + 2 * 2 + 2 * kRing + 2 * 2;
    static constexpr size_t tmem_slot() { return bars() + kNumBars * 8; }
    static constexpr size_t total() { return tmem_slot() + 16 + 1024; }
};
static_assert(Smem::total() <= 227 * 1024, "shared memory budget");
static_assert(kRawBytes % 1024 == 0 && kWMinBytes % 1024 == 0, "atoms stay 1024-byte aligned");
static_assert(Smem::total() < (1u << 18), "descriptor start addresses stay inside their 14-bit field");

struct Bars {
    uint64_t *full, *empty;           // [kStages]: activations (TMA) + weights (converters)
    uint64_t *raw_full, *raw_empty;   // [kRawSlots]
    uint64_t *min_full, *min_empty;   // [2]: s8 tile (TMA) and mins (converters)
    uint64_t *sb_full, *sb_empty;     // [kRing]: X and Mn of a super-block
    uint64_t *dd_full, *dd_free;      // [2]
};

struct SmallParams {
    int N, K, B, nb;
    int splits;
    size_t split_stride;   // floats between two splits' partial sums
    const float *tscale;   // [B]
    float *y;              // [B][N], or [splits][split_stride] partials
    unsigned int *status;
};

__global__ void __maxnreg__(128)
q4k_gemm_small_kernel(const __grid_constant__ CUtensorMap tmap_hi, const __grid_constant__ CUtensorMap tmap_lo,
                      const __grid_constant__ CUtensorMap tmap_s, const __grid_constant__ CUtensorMap tmap_w,
                      const SmallParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    __shared__ volatile int abort_s;

    uint64_t *bm = reinterpret_cast<uint64_t *>(sm + Smem::bars());
    Bars bar;
    bar.full = bm;
    bar.empty = bar.full + kStages;
    bar.raw_full = bar.empty + kStages;
    bar.raw_empty = bar.raw_full + kRawSlots;
    bar.min_full = bar.raw_empty + kRawSlots;
    bar.min_empty = bar.min_full + 2;
    bar.sb_full = bar.min_empty + 2;
    bar.sb_empty = bar.sb_full + kRing;
    bar.dd_full = bar.sb_empty + kRing;
    bar.dd_free = bar.dd_full + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + Smem::tmem_slot());

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int split = blockIdx.x % p.splits;
    const int n0 = (blockIdx.x / p.splits) * SR;
    const int b_begin = (int)((long long)split * p.nb / p.splits);
    const int nb = (int)((long long)(split + 1) * p.nb / p.splits) - b_begin;
    const int nq = 2 * nb;   // operand stages (K = 128 each)

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bar.full[s], 1 + kConvWarps);
            mbar_init(&bar.empty[s], 1);
        }
        for (int s = 0; s < kRawSlots; ++s) {
            mbar_init(&bar.raw_full[s], 1);
            mbar_init(&bar.raw_empty[s], kConvWarps);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar.min_full[i], 1 + kConvWarps);
            mbar_init(&bar.min_empty[i], 1);
            mbar_init(&bar.dd_full[i], kConvWarps);
            mbar_init(&bar.dd_free[i], kEpiWarps);
        }
        for (int i = 0; i < kRing; ++i) {
            mbar_init(&bar.sb_full[i], 1);
            mbar_init(&bar.sb_empty[i], kEpiWarps);
        }
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
            prefetch_tmap(&tmap_hi);
            prefetch_tmap(&tmap_lo);
            prefetch_tmap(&tmap_s);
            prefetch_tmap(&tmap_w);
            bool ok = true;
            int next_raw = 0;
            auto load_raw = [&](int bb) -> bool {
                const int rs = bb % kRawSlots, use = bb / kRawSlots;
                if (use > 0 && !wait_fast(&bar.raw_empty[rs], (use - 1) & 1, &abort_s, p.status)) return false;
                mbar_arrive_expect_tx(&bar.raw_full[rs], kRawBytes);
                tma_load_2d(sm + Smem::raw(rs), &tmap_w, kQ4KBlockBytes * (b_begin + bb), n0, &bar.raw_full[rs]);
                return true;
            };
            for (; next_raw < nb && next_raw < kRawSlots - 1 && ok; ++next_raw) ok = load_raw(next_raw);
            for (int q = 0; q < nq && ok; ++q) {
                const int b = q >> 1, i = q & 1;
                if (i == 0 && next_raw < nb) {
                    if (!(ok = load_raw(next_raw))) break;
                    ++next_raw;
                }
                const int s = q % kStages, round = q / kStages;
                if (round > 0 && !(ok = wait_fast(&bar.empty[s], (round - 1) & 1, &abort_s, p.status))) break;
                const int kx = 256 * (b_begin + b) + 128 * i;
                uint8_t *as = sm + Smem::a_stage(s);
                mbar_arrive_expect_tx(&bar.full[s], kAStageBytes);
                tma_load_2d(as, &tmap_hi, kx, 0, &bar.full[s]);
                tma_load_2d(as + kAAtom, &tmap_lo, kx, 0, &bar.full[s]);
                tma_load_2d(as + 2 * kAAtom, &tmap_hi, kx + 64, 0, &bar.full[s]);
                tma_load_2d(as + 3 * kAAtom, &tmap_lo, kx + 64, 0, &bar.full[s]);
                if (i == 0) {
                    const int mi = b & 1, use = b >> 1;
                    if (use > 0 && !(ok = wait_fast(&bar.min_empty[mi], (use - 1) & 1, &abort_s, p.status))) break;
                    mbar_arrive_expect_tx(&bar.min_full[mi], kAMinBytes);
                    tma_load_2d(sm + Smem::amin(mi), &tmap_s, 8 * (b_begin + b), 0, &bar.min_full[mi]);
                }
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t base = smem_u32(sm);
            const uint64_t w_desc0 = smem_desc(base + (uint32_t)Smem::w_stage(0), 16, 1024, kLayoutSw128);
            const uint64_t a_desc0 = smem_desc(base + (uint32_t)Smem::a_stage(0), 16, 1024, kLayoutSw128);
            const uint64_t wmin_desc0 = smem_desc(base + (uint32_t)Smem::wmin(0), 16, 256, kLayoutSw32);
            const uint64_t amin_desc0 = smem_desc(base + (uint32_t)Smem::amin(0), 16, 256, kLayoutSw32);
            constexpr uint32_t kW16 = kWAtom >> 4, kA16 = kAAtom >> 4;
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int b = 0; b < nb && ok; ++b) {
                const int slot = b % kRing, mi = b & 1;
                const uint32_t use = (uint32_t)(b / kRing);
                const uint32_t x_tmem = tmem + (uint32_t)(kSlotCols * slot), m_tmem = x_tmem + 2 * ST;
                if (use > 0 && !(ok = wait_fast(&bar.sb_empty[slot], (use - 1) & 1, &abort_s, p.status))) break;
                tc_fence_after();
                for (int i = 0; i < 2; ++i) {
                    if (!(ok = wait_fast(&bar.full[s], ph, &abort_s, p.status))) break;
                    tc_fence_after();
                    const uint64_t wd = w_desc0 + (uint64_t)(s * (kWStageBytes >> 4));
                    const uint64_t ad = a_desc0 + (uint64_t)(s * (kAStageBytes >> 4));
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_f16(x_tmem, wd + (uint64_t)(c * kW16 + 2 * kk),
                                    ad + (uint64_t)(2 * c * kA16 + 2 * kk), kIdesc, (i | c | kk) != 0 ? 1u : 0u);
                    }
                    mma_commit(&bar.empty[s]);
                    if (++s == kStages) { s = 0; ph ^= 1u; }
                }
                if (!ok) break;
                // the super-block's min product: sum_j m_j[n] * s8[t][bj]
                if (!(ok = wait_fast(&bar.min_full[mi], (uint32_t)(b >> 1) & 1, &abort_s, p.status))) break;
                tc_fence_after();
                mma_f16(m_tmem, wmin_desc0 + (uint64_t)(mi * (kWMinBytes >> 4)),
                        amin_desc0 + (uint64_t)(mi * (kAMinBytes >> 4)), kIdescMin, 0u);
                mma_commit(&bar.sb_full[slot]);
                mma_commit(&bar.min_empty[mi]);
            }
        }
    } else if (warp < kEpiWarp0) {
        // ---------------------------------------------------- converters
        // thread (r, h) converts nibble bytes 16h .. 16h+15 of each 32-byte
        // group of row r: weights 16h.. of the group's two sub-blocks
        const int ct = (warp - kConvWarp0) * 32 + lane;
        const int r = ct & (SR - 1), h = ct >> 7;
        const int sw = r & 7;
        for (int b = 0; b < nb; ++b) {
            const int rs = b % kRawSlots, ruse = b / kRawSlots;
            if (!warp_wait(&bar.raw_full[rs], ruse & 1, &abort_s, p.status)) break;
            const uint8_t *raw = sm + Smem::raw(rs) + (size_t)r * kQ4KBlockBytes;
            const uint4 hdr = *reinterpret_cast<const uint4 *>(raw);
            bool ok = true;
            for (int i = 0; i < 2 && ok; ++i) {
                const int q = 2 * b + i;
                const int s = q % kStages, round = q / kStages;
                if (round > 0 && !(ok = warp_wait(&bar.empty[s], (round - 1) & 1, &abort_s, p.status))) break;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int g = 2 * i + c;   // nibble group: sub-blocks 2g (low), 2g+1 (high)
                    const uint4 nv = *reinterpret_cast<const uint4 *>(raw + 16 + 32 * g + 16 * h);
                    uint32_t sc0, sc1, md;
                    q4k_scale_min(hdr.y, hdr.z, hdr.w, 2 * g, sc0, md);
                    q4k_scale_min(hdr.y, hdr.z, hdr.w, 2 * g + 1, sc1, md);
                    const float scl = (float)sc0, sch = (float)sc1;
                    const __half2 s_lo = __float2half2_rn(scl), o_lo = __float2half2_rn(-1024.0f * scl);
                    const __half2 s_hi = __float2half2_rn(sch * 0.0625f), o_hi = __float2half2_rn(-64.0f * sch);
                    const uint32_t wv[4] = {nv.x, nv.y, nv.z, nv.w};
                    uint8_t *atom = sm + Smem::w_stage(s) + (size_t)c * kWAtom + (size_t)r * 128;
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        uint4 lo, hi;
                        nib4_to_h2<false>(wv[2 * u], s_lo, o_lo, lo.x, lo.y);
                        nib4_to_h2<false>(wv[2 * u + 1], s_lo, o_lo, lo.z, lo.w);
                        nib4_to_h2<true>(wv[2 * u], s_hi, o_hi, hi.x, hi.y);
                        nib4_to_h2<true>(wv[2 * u + 1], s_hi, o_hi, hi.z, hi.w);
                        const int cl = 2 * h + u;   // 16-byte chunk of the 128-byte row
                        *reinterpret_cast<uint4 *>(atom + ((cl ^ sw) << 4)) = lo;
                        *reinterpret_cast<uint4 *>(atom + (((cl + 4) ^ sw) << 4)) = hi;
                    }
                }
                if (i == 0) {
                    const int mi = b & 1, use = b >> 1;
                    if (use > 0 && !(ok = warp_wait(&bar.min_empty[mi], (use - 1) & 1, &abort_s, p.status))) break;
                    if (use > 0 && !(ok = warp_wait(&bar.dd_free[mi], (use - 1) & 1, &abort_s, p.status))) break;
                    if (h == 0) {
                        uint32_t mn[8], scd;
#pragma unroll
                        for (int j = 0; j < 8; ++j) q4k_scale_min(hdr.y, hdr.z, hdr.w, j, scd, mn[j]);
                        uint4 m0;
                        m0.x = h2_bits(__floats2half2_rn((float)mn[0], (float)mn[1]));
                        m0.y = h2_bits(__floats2half2_rn((float)mn[2], (float)mn[3]));
                        m0.z = h2_bits(__floats2half2_rn((float)mn[4], (float)mn[5]));
                        m0.w = h2_bits(__floats2half2_rn((float)mn[6], (float)mn[7]));
                        uint8_t *bmr = sm + Smem::wmin(mi) + (size_t)r * 32;
                        const int s32 = (r >> 2) & 1;
                        *reinterpret_cast<uint4 *>(bmr + ((0 ^ s32) << 4)) = m0;
                        *reinterpret_cast<uint4 *>(bmr + ((1 ^ s32) << 4)) = make_uint4(0, 0, 0, 0);
                        const float2 dm = __half22float2(*reinterpret_cast<const __half2 *>(&hdr.x));
                        float *ddp = reinterpret_cast<float *>(sm + Smem::dd(mi));
                        ddp[r] = dm.x;
                        ddp[SR + r] = -dm.y;
                    }
                    fence_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&bar.min_full[mi]);
                        mbar_arrive(&bar.dd_full[mi]);
                    }
                }
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar.full[s]);
            }
            if (!ok) break;
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar.raw_empty[rs]);
        }
    } else {
        // ---------------------------------------------------- epilogue
        const int quarter = warp & 3;                 // TMEM lanes 32*quarter .. +31
        const int row = 32 * quarter + lane;          // weight row within the tile
        const uint32_t lane_base = tmem + ((uint32_t)(32 * quarter) << 16);
        float tsc[ST], itsc[ST], acc[ST];
#pragma unroll
        for (int t = 0; t < ST; ++t) {
            tsc[t] = t < p.B ? p.tscale[t] : 1.0f;
            itsc[t] = 1.0f / tsc[t];   // exact: a power of two
            acc[t] = 0.0f;
        }
        bool ok = true;
        for (int b = 0; b < nb && ok; ++b) {
            const int slot = b % kRing, mi = b & 1;
            if (!(ok = warp_wait(&bar.dd_full[mi], (uint32_t)(b >> 1) & 1, &abort_s, p.status))) break;
            if (!(ok = warp_wait(&bar.sb_full[slot], (uint32_t)(b / kRing) & 1, &abort_s, p.status))) break;
            tc_fence_after();
            uint32_t xr[16], xl[16], mr[16];
            tmem_ld16(lane_base + (uint32_t)(kSlotCols * slot), xr);
            tmem_ld16(lane_base + (uint32_t)(kSlotCols * slot + ST), xl);
            tmem_ld16(lane_base + (uint32_t)(kSlotCols * slot + 2 * ST), mr);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar.sb_empty[slot]);
            const float *ddp = reinterpret_cast<const float *>(sm + Smem::dd(mi));
            const float d = ddp[row], ndm = ddp[SR + row];
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar.dd_free[mi]);
#pragma unroll
            for (int t = 0; t < ST; ++t) {
                acc[t] = fmaf(d, __uint_as_float(xr[t]), acc[t]);
                acc[t] = fmaf(d, __uint_as_float(xl[t]), acc[t]);
                acc[t] = fmaf(ndm * itsc[t], __uint_as_float(mr[t]), acc[t]);
            }
        }
        if (ok && !abort_s && n0 + row < p.N) {
            float *yc = p.y + (size_t)split * p.split_stride + n0 + row;
#pragma unroll
            for (int t = 0; t < ST; ++t)
                if (t < p.B) yc[(size_t)t * p.N] = acc[t] * tsc[t];
        }
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

size_t g_attr_bytes[64];

}  // namespace

cudaError_t launch_gemm_small(const void *W, int N, int K, int B, const __half *hi, const __half *lo,
                              const __half *s8, const float *tscale, float *out, float *y, int splits,
                              cudaStream_t st)
{
    CUtensorMap th, tl, ts, tw;
    const CUtensorMapDataType f16 = CU_TENSOR_MAP_DATA_TYPE_FLOAT16, u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
    cudaError_t e;
    // token rows beyond B read as zero (out-of-range box rows)
    if ((e = make_tmap_2d(&th, f16, 2, hi, (uint64_t)K, (uint64_t)B, 64, ST, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
        return e;
    if ((e = make_tmap_2d(&tl, f16, 2, lo, (uint64_t)K, (uint64_t)B, 64, ST, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
        return e;
    if ((e = make_tmap_2d(&ts, f16, 2, s8, (uint64_t)K / 32, (uint64_t)B, 16, ST, CU_TENSOR_MAP_SWIZZLE_32B)) !=
        cudaSuccess)
        return e;
    if ((e = make_tmap_2d(&tw, u8, 1, W, (uint64_t)(K / 256) * kQ4KBlockBytes, (uint64_t)N, kQ4KBlockBytes, SR,
                          CU_TENSOR_MAP_SWIZZLE_NONE)) != cudaSuccess)
        return e;
    SmallParams p{};
    p.N = N;
    p.K = K;
    p.B = B;
    p.nb = K / 256;
    p.splits = splits;
    p.split_stride = split_stride(B, N);
    p.tscale = tscale;
    p.y = out;
    p.status = device_status_word();
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    const size_t smem = Smem::total();
    if (g_attr_bytes[dev] < smem) {
        e = cudaFuncSetAttribute(q4k_gemm_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        g_attr_bytes[dev] = smem;
    }
    const long long grid = (long long)((N + SR - 1) / SR) * splits;
    q4k_gemm_small_kernel<<<(unsigned)grid, kThreads, smem, st>>>(th, tl, ts, tw, p);
    if (splits == 1) return cudaGetLastError();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    return launch_splitk_reduce(out, splits, (size_t)B * N, y, st);
}

}  // namespace zq
