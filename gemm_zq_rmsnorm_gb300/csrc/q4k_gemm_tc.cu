// q4k_gemm_tc.cu -- batched Q4_K x Q8_1 projection on the tcgen05 tensor
// cores (B >= 2 tokens).
//
// MIInfer README, "Current phase": token-batched chunk projections for
// prefill and tensor-core prefill; ZINC docs "ROCm backend", "Build and
// verify": matrix-core prefill tiles that consume the Q4 weights directly.
//
// The projection is
//   y[t][n] = sum_b d_b[n] * sum_{k in b} x'[t][k] * w[n][k]
//           - sum_b dmin_b[n] * sum_j m_j[n] * s8[t][bj],
// with x'[t][k] = q8[t][k] * d8[t][k/32] (the Q8_1 value) and w = sc_j * q4,
// an integer up to 945.  sm_103a has no int8 tcgen05 MMA, and scaling 32-wide
// integer partial sums by d8 one sub-block at a time makes the epilogue, not
// the tensor cores, the bound.  Instead every x' (18 significant bits, exact in
// fp32) is split into two binary16 numbers, hi = fp16(x') and lo = fp16(x' - hi)
// (at most 7 significant bits, exact), and each K = 16 step issues two MMAs,
// hi * w and lo * w, into one fp32 accumulator.  Every product is exact; the
// only rounding is the fp32 accumulation over the 256 weights of a
// super-block.  Tokens whose codes would overflow binary16 are scaled by a
// power of two first (undone exactly in the epilogue).  So one TMEM
// accumulator per super-block replaces eight per-sub-block ones: the epilogue
// folds it in with acc += d_b * X once per super-block, and a small MMA per
// super-block forms the min term sum_j s8[t][bj] * m_j[n] (s8 a binary16
// value, m_j <= 63: exact products) that it subtracts as dmin_b * Mn.
//
// Tile: M = 128 tokens (TMEM lanes) x N = 128 weight rows (TMEM columns).
// TMEM (512 columns) holds two super-blocks in flight, each an X and an Mn
// buffer.  Warp roles (26 warps): 0 TMA producer (hi/lo activation tiles and
// s8 tiles, raw Q4_K tiles two super-blocks ahead), 1 MMA issuer + TMEM owner,
// 2-9 weight converters (Q4_K bytes -> sc*q fp16 in the 128-byte-swizzled
// K-major layout, half a row per thread; mins; d/dmin), 10-25 epilogue (4
// column groups of 32 x 4 lane quarters) holding the fp32 accumulator in
// registers.
// Every wait is bounded.
#include <cuda.h>

#include "zq_internal.cuh"
#include "zq_tc.cuh"
#include "zq_tc_common.cuh"

namespace zq {
namespace {

constexpr int BM = 128;               // tokens per tile (TMEM lanes)
constexpr int BN = 128;               // weight rows per tile (TMEM columns)
constexpr int kStages = 3;            // operand stages of K = 64 (two sub-blocks)
constexpr int kAtomBytes = 128 * 128; // 128 rows x 64 fp16 (128 B), 128-byte swizzle
constexpr int kAStageBytes = 2 * kAtomBytes;    // hi atom, lo atom
constexpr int kRawSlots = 3;          // raw Q4_K tiles in flight (super-blocks)
constexpr int kRawBytes = BN * kQ4KBlockBytes;  // 128 rows x 144 B
constexpr int kMinBytes = 128 * 32;   // 128 rows x 16 fp16, 32-byte swizzle
constexpr int kWarps = 26;
constexpr int kThreads = kWarps * 32;
constexpr int kConvWarp0 = 2, kConvWarps = 8;   // a converter thread owns half of one weight row
constexpr int kEpiWarp0 = 10, kEpiWarps = 16;
constexpr int kEpiCols = BN / (kEpiWarps / 4);   // 32 columns per epilogue thread
// registers: warps are spread over the SM's four sub-partitions, at most
// ceil(26 / 4) = 7 on one, and a sub-partition holds 16384 registers
constexpr int kMaxRegs = 72;
static_assert(((kWarps + 3) / 4) * 32 * kMaxRegs <= 16384, "register file of one sub-partition");
static_assert(kConvWarps * 32 == 2 * BN, "two converter threads per weight row");
static_assert(kEpiWarp0 % 4 == 2, "epilogue lane quarters follow warp % 4");
constexpr uint32_t kIdesc = idesc_f16_f32(BM, BN);
constexpr uint32_t kTmemCols = 512;   // [X0 | Mn0 | X1 | Mn1], 128 columns each

struct Smem {
    // offsets from the 1024-aligned base
    static constexpr size_t a_stage(int s) { return (size_t)s * kAStageBytes; }  // hi, then lo
    static constexpr size_t b_atom(int s) { return a_stage(kStages) + (size_t)s * kAtomBytes; }
    static constexpr size_t raw(int i) { return b_atom(kStages) + (size_t)i * kRawBytes; }
    static constexpr size_t amin(int i) { return raw(kRawSlots) + (size_t)i * 2 * kMinBytes; }
    static constexpr size_t bmin(int i) { return amin(i) + kMinBytes; }
    static constexpr size_t dd(int i) { return amin(2) + (size_t)i * BN * 8; }  // d[BN], then -dmin[BN]
    static constexpr size_t bars() { return dd(2); }
    static constexpr int kNumBars = 2 * kStages + 2 * kRawSlots + 2 * 2 + 2 * 4 + 2 * 2;
    static constexpr size_t tmem_slot() { return bars() + kNumBars * 8; }
    static constexpr size_t total() { return tmem_slot() + 16 + 1024; }  // + alignment slack
};
static_assert(Smem::total() <= 227 * 1024, "shared memory budget");
static_assert(kRawBytes % 1024 == 0, "raw slots keep the operand atoms 1024-byte aligned");
static_assert(Smem::total() < (1u << 18), "descriptor start addresses stay inside their 14-bit field");

struct Bars {
    // full[s]: the TMA's activation bytes and every converter warp's weights
    // of stage s have landed (one wait for the issuer); empty[s]: the MMAs
    // reading stage s have completed
    uint64_t *full, *empty;                       // [kStages]
    uint64_t *raw_full, *raw_empty;               // [kRawSlots]
    uint64_t *min_full, *min_empty;               // [2]: s8 tile (TMA) and mins (converters)
    uint64_t *ring_full, *ring_empty;             // [4]: X0, Mn0, X1, Mn1
    uint64_t *dd_full, *dd_free;                  // [2]
};

struct GemmParams {
    int N, K, B, nb;
    int t_tiles;
    int splits;            // K ranges (split-K); CTA = (split, token tile, weight tile)
    size_t split_stride;   // floats between two splits' partial sums (split_stride(B, N))
    const float *tscale;   // [B] power of two that undoes the code scaling
    float *y;              // [B][N], or [splits][split_stride] partial sums when splits > 1
    unsigned int *status;
};

// (c0, c1) += (a0, a1) * (b0, b1)
__device__ __forceinline__ void fma2(float &c0, float &c1, float a0, float a1, float b0, float b1)
{
    asm("{\n\t.reg .b64 ra, rb, rc;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%0, %1};\n\t"
        "fma.rn.f32x2 rc, ra, rb, rc;\n\tmov.b64 {%0, %1}, rc;\n\t}"
        : "+f"(c0), "+f"(c1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

__global__ void __maxnreg__(kMaxRegs)
q4k_gemm_tc_kernel(const __grid_constant__ CUtensorMap tmap_hi, const __grid_constant__ CUtensorMap tmap_lo,
                   const __grid_constant__ CUtensorMap tmap_s, const __grid_constant__ CUtensorMap tmap_w,
                   const GemmParams p)
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
    bar.ring_full = bar.min_empty + 2;
    bar.ring_empty = bar.ring_full + 4;
    bar.dd_full = bar.ring_empty + 4;
    bar.dd_free = bar.dd_full + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + Smem::tmem_slot());

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int split = blockIdx.x % p.splits;
    const int tile = blockIdx.x / p.splits;
    const int t_tile = tile % p.t_tiles;
    const int n_tile = tile / p.t_tiles;
    const int t0 = t_tile * BM;
    const int n0 = n_tile * BN;
    // this CTA's super-blocks: [b_begin, b_begin + nb) of the row
    const int b_begin = (int)((long long)split * p.nb / p.splits);
    const int nb = (int)((long long)(split + 1) * p.nb / p.splits) - b_begin;
    const int nq = 4 * nb;   // operand stages (K = 64 each)
    // Each CTA walks its super-blocks in its own rotated order, so the CTAs
    // that share an activation tile (and those that share a weight tile) do not
    // all request the same L2 lines at the same time.
    const int rot = (n_tile + 5 * t_tile) % nb;
    auto sb = [&](int b) { return b_begin + (b + rot < nb ? b + rot : b + rot - nb); };

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
        for (int i = 0; i < 4; ++i) {
            mbar_init(&bar.ring_full[i], 1);
            mbar_init(&bar.ring_empty[i], kEpiWarps);
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
            // raw weight tiles run kRawSlots - 1 super-blocks ahead of the
            // activation tiles; stage q = 4b + i
            int next_raw = 0;
            auto load_raw = [&](int bb) -> bool {
                const int rs = bb % kRawSlots, use = bb / kRawSlots;
                if (use > 0 && !wait_fast(&bar.raw_empty[rs], (use - 1) & 1, &abort_s, p.status)) return false;
                mbar_arrive_expect_tx(&bar.raw_full[rs], kRawBytes);
                tma_load_2d(sm + Smem::raw(rs), &tmap_w, kQ4KBlockBytes * sb(bb), n0, &bar.raw_full[rs]);
                return true;
            };
            for (; next_raw < nb && next_raw < kRawSlots - 1 && ok; ++next_raw) ok = load_raw(next_raw);
            for (int q = 0; q < nq && ok; ++q) {
                const int b = q >> 2, i = q & 3;
                if (i == 0 && next_raw < nb) {
                    if (!(ok = load_raw(next_raw))) break;
                    ++next_raw;
                }
                const int s = q % kStages, round = q / kStages;
                if (round > 0 && !(ok = wait_fast(&bar.empty[s], (round - 1) & 1, &abort_s, p.status))) break;
                const int kx = 256 * sb(b) + 64 * i;
                mbar_arrive_expect_tx(&bar.full[s], kAStageBytes);
                tma_load_2d(sm + Smem::a_stage(s), &tmap_hi, kx, t0, &bar.full[s]);
                tma_load_2d(sm + Smem::a_stage(s) + kAtomBytes, &tmap_lo, kx, t0, &bar.full[s]);
                if (i == 0) {
                    const int mi = b & 1, use = b >> 1;
                    if (use > 0 && !(ok = wait_fast(&bar.min_empty[mi], (use - 1) & 1, &abort_s, p.status))) break;
                    mbar_arrive_expect_tx(&bar.min_full[mi], kMinBytes);
                    tma_load_2d(sm + Smem::amin(mi), &tmap_s, 8 * sb(b), t0, &bar.min_full[mi]);
                }
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t base = smem_u32(sm);
            // descriptors of stage 0 / min slot 0; every other operand tile is
            // reached by adding its byte offset / 16 to the start-address field
            const uint64_t a_desc0 = smem_desc(base + (uint32_t)Smem::a_stage(0), 16, 1024, kLayoutSw128);
            const uint64_t b_desc0 = smem_desc(base + (uint32_t)Smem::b_atom(0), 16, 1024, kLayoutSw128);
            const uint64_t amin_desc0 = smem_desc(base + (uint32_t)Smem::amin(0), 16, 256, kLayoutSw32);
            const uint64_t bmin_desc0 = smem_desc(base + (uint32_t)Smem::bmin(0), 16, 256, kLayoutSw32);
            constexpr uint32_t kAtom16 = kAtomBytes >> 4, kMinSlot16 = (2 * kMinBytes) >> 4;
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int b = 0; b < nb && ok; ++b) {
                const int mi = b & 1;
                const uint32_t use = (uint32_t)(b >> 1);   // earlier super-blocks on these buffers
                const uint32_t xbuf = 2u * (uint32_t)mi, mbuf = xbuf + 1u;
                const uint32_t x_tmem = tmem + (uint32_t)BN * xbuf;
                if (use > 0 && !(ok = wait_fast(&bar.ring_empty[xbuf], (use - 1) & 1, &abort_s, p.status))) break;
                tc_fence_after();
                for (int i = 0; i < 4; ++i) {
                    if (!(ok = wait_fast(&bar.full[s], ph, &abort_s, p.status))) break;
                    tc_fence_after();
                    const uint64_t ahi = a_desc0 + (uint64_t)(2 * s * kAtom16);
                    const uint64_t alo = ahi + (uint64_t)kAtom16;
                    const uint64_t bd = b_desc0 + (uint64_t)(s * kAtom16);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        mma_f16(x_tmem, ahi + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk), kIdesc,
                                (i | kk) != 0 ? 1u : 0u);
                        mma_f16(x_tmem, alo + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk), kIdesc, 1u);
                    }
                    mma_commit(&bar.empty[s]);
                    if (++s == kStages) { s = 0; ph ^= 1u; }
                }
                if (!ok) break;
                mma_commit(&bar.ring_full[xbuf]);
                // the super-block's min product: sum_j s8[t][bj] * m_j[n]
                if (!(ok = wait_fast(&bar.min_full[mi], use & 1, &abort_s, p.status) &&
                           (use == 0 || wait_fast(&bar.ring_empty[mbuf], (use - 1) & 1, &abort_s, p.status))))
                    break;
                tc_fence_after();
                mma_f16(tmem + (uint32_t)BN * mbuf, amin_desc0 + (uint64_t)(mi * kMinSlot16),
                        bmin_desc0 + (uint64_t)(mi * kMinSlot16), kIdesc, 0u);
                mma_commit(&bar.ring_full[mbuf]);
                mma_commit(&bar.min_empty[mi]);
            }
        }
    } else if (warp < kEpiWarp0) {
        // ---------------------------------------------------- converters
        // thread (r, h) converts bytes 16h .. 16h+15 of weight row r's 32-byte
        // nibble group: weights 16h.. of the stage's first sub-block (low
        // nibbles) and of its second (high nibbles); h = 0 also writes the
        // row's mins and d / -dmin once per super-block
        const int ct = (warp - kConvWarp0) * 32 + lane;
        const int r = ct & (BN - 1), h = ct >> 7;
        const int sw = r & 7;
        for (int b = 0; b < nb; ++b) {
            const int rs = b % kRawSlots, ruse = b / kRawSlots;
            if (!warp_wait(&bar.raw_full[rs], ruse & 1, &abort_s, p.status)) break;
            const uint8_t *raw = sm + Smem::raw(rs) + (size_t)r * kQ4KBlockBytes;
            const uint4 hdr = *reinterpret_cast<const uint4 *>(raw);
            bool ok = true;
            for (int i = 0; i < 4 && ok; ++i) {
                const int q = 4 * b + i;
                const int s = q % kStages, round = q / kStages;
                if (round > 0 && !(ok = warp_wait(&bar.empty[s], (round - 1) & 1, &abort_s, p.status))) break;
                const uint4 nv = *reinterpret_cast<const uint4 *>(raw + 16 + 32 * i + 16 * h);
                uint32_t sc0, sc1, md;
                q4k_scale_min(hdr.y, hdr.z, hdr.w, 2 * i, sc0, md);
                q4k_scale_min(hdr.y, hdr.z, hdr.w, 2 * i + 1, sc1, md);
                const float scl = (float)sc0, sch = (float)sc1;
                const __half2 s_lo = __float2half2_rn(scl), o_lo = __float2half2_rn(-1024.0f * scl);
                const __half2 s_hi = __float2half2_rn(sch * 0.0625f), o_hi = __float2half2_rn(-64.0f * sch);
                const uint32_t wv[4] = {nv.x, nv.y, nv.z, nv.w};
                uint8_t *atom = sm + Smem::b_atom(s) + (size_t)r * 128;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint4 lo, hi;
                    nib4_to_h2<false>(wv[2 * c], s_lo, o_lo, lo.x, lo.y);
                    nib4_to_h2<false>(wv[2 * c + 1], s_lo, o_lo, lo.z, lo.w);
                    nib4_to_h2<true>(wv[2 * c], s_hi, o_hi, hi.x, hi.y);
                    nib4_to_h2<true>(wv[2 * c + 1], s_hi, o_hi, hi.z, hi.w);
                    const int cl = 2 * h + c;   // 16-byte chunk of the 128-byte row
                    *reinterpret_cast<uint4 *>(atom + ((cl ^ sw) << 4)) = lo;
                    *reinterpret_cast<uint4 *>(atom + (((cl + 4) ^ sw) << 4)) = hi;
                }
                if (i == 0) {
                    const int mi = b & 1, use = b >> 1;
                    // mins as the B operand of the min MMA; d, -dmin for the epilogue
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
                        uint8_t *bmr = sm + Smem::bmin(mi) + (size_t)r * 32;
                        const int s32 = (r >> 2) & 1;
                        *reinterpret_cast<uint4 *>(bmr + ((0 ^ s32) << 4)) = m0;
                        *reinterpret_cast<uint4 *>(bmr + ((1 ^ s32) << 4)) = make_uint4(0, 0, 0, 0);
                        const float2 dm = __half22float2(*reinterpret_cast<const __half2 *>(&hdr.x));
                        float *ddp = reinterpret_cast<float *>(sm + Smem::dd(mi));
                        ddp[r] = dm.x;
                        ddp[BN + r] = -dm.y;
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
        const int e_w = warp - kEpiWarp0;
        const int cg = e_w >> 2;                  // column group: columns 64cg .. 64cg+63
        const int quarter = warp & 3;             // TMEM lanes 32*quarter .. +31
        const int tok = t0 + 32 * quarter + lane;
        const bool tvalid = tok < p.B;
        const uint32_t lane_base = tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(kEpiCols * cg);
        // X carries the codes' scale 2^-k; scale the min term the same way and
        // undo both at the store
        const float tsc = tvalid ? p.tscale[tok] : 1.0f;
        const float itsc = 1.0f / tsc;   // exact: tsc is a power of two
        float acc[kEpiCols];
#pragma unroll
        for (int c = 0; c < kEpiCols; ++c) acc[c] = 0.0f;
        bool ok = true;
        for (int b = 0; b < nb && ok; ++b) {
            const int mi = b & 1;
            const uint32_t use = (uint32_t)(b >> 1);
            const uint32_t xbuf = 2u * (uint32_t)mi, mbuf = xbuf + 1u;
            if (!(ok = warp_wait(&bar.dd_full[mi], use & 1, &abort_s, p.status))) break;
            const float *dcol = reinterpret_cast<const float *>(sm + Smem::dd(mi)) + kEpiCols * cg;
            uint32_t r[16];
            // acc += d_b * X, 16 columns at a time
            if (!(ok = warp_wait(&bar.ring_full[xbuf], use & 1, &abort_s, p.status))) break;
            tc_fence_after();
#pragma unroll
            for (int q = 0; q < kEpiCols / 16; ++q) {
                tmem_ld16(lane_base + (uint32_t)BN * xbuf + 16u * q, r);
                tmem_wait_ld();
                if (q == kEpiCols / 16 - 1) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bar.ring_empty[xbuf]);
                }
#pragma unroll
                for (int c = 0; c < 16; c += 2) {
                    const float2 dv = *reinterpret_cast<const float2 *>(dcol + 16 * q + c);
                    fma2(acc[16 * q + c], acc[16 * q + c + 1], dv.x, dv.y, __uint_as_float(r[c]),
                         __uint_as_float(r[c + 1]));
                }
            }
            // acc -= dmin_b * Mn * 2^-k
            if (!(ok = warp_wait(&bar.ring_full[mbuf], use & 1, &abort_s, p.status))) break;
            tc_fence_after();
#pragma unroll
            for (int q = 0; q < kEpiCols / 16; ++q) {
                tmem_ld16(lane_base + (uint32_t)BN * mbuf + 16u * q, r);
                tmem_wait_ld();
                if (q == kEpiCols / 16 - 1) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bar.ring_empty[mbuf]);
                }
#pragma unroll
                for (int c = 0; c < 16; c += 2) {
                    const float2 mv = *reinterpret_cast<const float2 *>(dcol + BN + 16 * q + c);
                    fma2(acc[16 * q + c], acc[16 * q + c + 1], mv.x * itsc, mv.y * itsc, __uint_as_float(r[c]),
                         __uint_as_float(r[c + 1]));
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar.dd_free[mi]);
        }
        if (ok && !abort_s && tvalid) {
            const int sp_now = (int)(blockIdx.x % (unsigned)p.splits);
            float *yrow = p.y + (size_t)sp_now * p.split_stride + (size_t)tok * p.N + n0 + kEpiCols * cg;
            const int ncols = min(kEpiCols, p.N - (n0 + kEpiCols * cg));
            if (ncols == kEpiCols && (p.N & 3) == 0) {
#pragma unroll
                for (int c = 0; c < kEpiCols; c += 4)
                    *reinterpret_cast<float4 *>(yrow + c) =
                        make_float4(acc[c] * tsc, acc[c + 1] * tsc, acc[c + 2] * tsc, acc[c + 3] * tsc);
            } else {
#pragma unroll
                for (int c = 0; c < kEpiCols; ++c)
                    if (c < ncols) yrow[c] = acc[c] * tsc;
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

// One CTA per token: x' = q8 * d8 split into binary16 hi + lo.  The token's
// codes are scaled by 2^-k, k >= 0 the least that keeps 127 * max d8 within
// binary16 range, and tscale[t] = 2^k.
constexpr int kSplitThreads = 256;

__global__ void __launch_bounds__(kSplitThreads)
q8_split_kernel(const int8_t *__restrict__ qs, const __half *__restrict__ d8, int K, __half *__restrict__ hi,
                __half *__restrict__ lo, float *__restrict__ tscale)
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
    int k = 0;
    const float bound = 127.0f * m;   // >= every |x'| of the token
    if (bound > 65504.0f) frexpf(bound / 65504.0f, &k);   // bound / 65504 <= 2^k
    const float down = ldexpf(1.0f, -k);
    if (threadIdx.x == 0) tscale[t] = ldexpf(1.0f, k);
    const int8_t *qt = qs + (size_t)t * K;
    for (int g = threadIdx.x; g < (K >> 4); g += kSplitThreads) {
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
// partial sums [splits][split_stride(B, N)] fp32 (when splits > 1)
size_t split_bytes(int K, int B) { return (size_t)B * K * sizeof(__half); }
size_t tscale_bytes(int B) { return ((size_t)B * sizeof(float) + 255) & ~(size_t)255; }

// Split-K count: tiles that fill the SMs unevenly waste whole waves (a
// 512 x 5120 output is 160 tiles for 152 SMs: two waves, the second almost
// empty).  Model the time of `s` splits as waves * (super-blocks per split +
// a fixed per-CTA cost) plus the partial-sum traffic, and take the smallest
// s within 3 % of the best, keeping >= 2 super-blocks per split.
int choose_splits(int B, int N, int K, int sms)
{
    // both tensor-core kernels tile the weight rows by 128; the batched one
    // also tiles the tokens by 128, the small-batch one takes all B <= 16
    const long long tiles = (long long)((B + BM - 1) / BM) * ((N + BN - 1) / BN);
    const int nb = K / 256;
    const int smax = nb / 2 < 8 ? nb / 2 : 8;
    double cost[9];
    double best = 1e300;
    for (int sp = 1; sp <= (smax > 1 ? smax : 1); ++sp) {
        const long long ctas = tiles * sp;
        const double waves = (double)((ctas + sms - 1) / sms);
        double c = waves * ((double)nb / sp + 1.5);
        if (sp > 1) c += (double)(sp + 1) * B * N * 4.0 / 1.85e7;   // partials, in super-block times
        cost[sp] = c;
        if (c < best) best = c;
    }
    for (int sp = 1; sp <= (smax > 1 ? smax : 1); ++sp)
        if (cost[sp] <= best * 1.03) return sp;
    return 1;
}

cudaError_t launch_q8_split(zq_q8_1 a, int K, int B, __half *hi, __half *lo, float *tscale, cudaStream_t st)
{
    q8_split_kernel<<<B, kSplitThreads, 0, st>>>(a.qs, reinterpret_cast<const __half *>(a.d), K, hi, lo, tscale);
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

size_t gemm_tc_workspace_bytes(int N, int K, int B, bool allow_split)
{
    if (B <= 1) return 0;
    const int sp = allow_split ? choose_splits(B, N, K, num_sms()) : 1;
    return 2 * split_bytes(K, B) + tscale_bytes(B) + (sp > 1 ? (size_t)sp * split_stride(B, N) * sizeof(float) : 0);
}

cudaError_t launch_gemm_tc(const void *W, int N, int K, zq_q8_1 a, int B, float *y, void *ws, bool allow_split,
                           cudaStream_t st)
{
    uint8_t *w8 = static_cast<uint8_t *>(ws);
    __half *hi = reinterpret_cast<__half *>(w8);
    __half *lo = reinterpret_cast<__half *>(w8 + split_bytes(K, B));
    float *tscale = reinterpret_cast<float *>(w8 + 2 * split_bytes(K, B));
    const int splits = allow_split ? choose_splits(B, N, K, num_sms()) : 1;
    float *part = reinterpret_cast<float *>(w8 + 2 * split_bytes(K, B) + tscale_bytes(B));
    cudaError_t e = launch_q8_split(a, K, B, hi, lo, tscale, st);
    if (e != cudaSuccess) return e;
    if (B <= kSmallMaxB)
        return launch_gemm_small(W, N, K, B, hi, lo, reinterpret_cast<const __half *>(a.s), tscale,
                                 splits > 1 ? part : y, y, splits, st);
    CUtensorMap th, tl, ts, tw;
    const CUtensorMapDataType f16 = CU_TENSOR_MAP_DATA_TYPE_FLOAT16, u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
    if ((e = make_tmap_2d(&th, f16, 2, hi, (uint64_t)K, (uint64_t)B, 64, BM, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
        return e;
    if ((e = make_tmap_2d(&tl, f16, 2, lo, (uint64_t)K, (uint64_t)B, 64, BM, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
        return e;
    if ((e = make_tmap_2d(&ts, f16, 2, a.s, (uint64_t)K / 32, (uint64_t)B, 16, BM, CU_TENSOR_MAP_SWIZZLE_32B)) !=
        cudaSuccess)
        return e;
    // weights as bytes [N][K/256*144]: one box = one super-block of 128 rows
    if ((e = make_tmap_2d(&tw, u8, 1, W, (uint64_t)(K / 256) * kQ4KBlockBytes, (uint64_t)N, kQ4KBlockBytes, BN,
                          CU_TENSOR_MAP_SWIZZLE_NONE)) != cudaSuccess)
        return e;
    GemmParams p{};
    p.N = N;
    p.K = K;
    p.B = B;
    p.nb = K / 256;
    p.t_tiles = (B + BM - 1) / BM;
    p.splits = splits;
    p.split_stride = split_stride(B, N);
    p.tscale = tscale;
    p.y = splits > 1 ? part : y;
    p.status = device_status_word();
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    const size_t smem = Smem::total();
    if (g_attr_bytes[dev] < smem) {
        e = cudaFuncSetAttribute(q4k_gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        g_attr_bytes[dev] = smem;
    }
    const long long grid = (long long)p.t_tiles * ((N + BN - 1) / BN) * splits;
    q4k_gemm_tc_kernel<<<(unsigned)grid, kThreads, smem, st>>>(th, tl, ts, tw, p);
    if (splits == 1) return cudaGetLastError();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    return launch_splitk_reduce(part, splits, (size_t)B * N, y, st);
}

}  // namespace zq
