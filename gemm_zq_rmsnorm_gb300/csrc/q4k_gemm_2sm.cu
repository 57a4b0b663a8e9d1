// q4k_gemm_2sm.cu -- batched Q4_K x Q8_1 projection (B >= 17 tokens) on the
// tensor cores of two SMs at a time (tcgen05 MMAs of a CTA pair).
//
// MIInfer README, "Current phase": tensor-core prefill that consumes the
// quantized weights directly (token-batched projections; int8 GEMM ceiling);
// ZINC docs "ROCm backend", "Build and verify": matrix-core prefill tiles.
//
// The projection is
//   y[t][n] = sum_b d_b[n] * ( sum_{k in b} x'[t][k] * w[n][k]
//                              - (dmin_b[n] / d_b[n]) * sum_j m_j[n] * s8[t][bj] ),
// x' = q8 * d8 (a Q8_1 value: 18 significant bits), w = sc_j * q4 (an integer
// up to 945, exact in binary16).  sm_103a has no int8 MMA; every x' is split
// into two binary16 numbers hi + lo (exact), and each K = 16 step issues
// hi * w and lo * w into one fp32 accumulator, so every product is exact and
// the only rounding is fp32 accumulation.  The min term of the super-block
// enters the same accumulator through one more K = 16 MMA: its A operand
// holds -(dmin/d) * m_j split into binary16 hi and lo parts (16 values per
// weight row), its B operand the token's eight s8 values twice.  So each
// super-block leaves one accumulator, X_b, that the epilogue folds into
// registers with acc += d_b * X_b.  (A weight row whose d is 0 uses dmin as
// the ratio and folds with 1; a ratio too large for binary16 is scaled by a
// power of two, undone in the fold.)
//
// Tile of a CTA pair: 256 weight rows (the MMA's M: 128 rows in each CTA's
// shared and tensor memory) x 256 tokens (the MMA's N: each CTA stages 128
// tokens, the MMA reads both halves).  Each CTA converts only its own 128
// weight rows, and every converted weight meets all 256 tokens; one
// 256 x 256 x 16 MMA keeps each SM's tensor core busy for ~128 cycles.
// Tensor memory (512 columns) holds two super-block accumulators of 256
// columns, so the MMAs of super-block b+1 run while the epilogue folds b.
//
// Warp roles (16 warps, four warpgroups):
//   0      TMA producer: raw Q4_K tiles (this CTA's 128 rows, two super-blocks
//          ahead), binary16 hi/lo token tiles and s8 tiles, whose bytes are
//          counted on the even CTA's stage barrier;
//   1      MMA issuer (even CTA only) and tensor-memory owner (both CTAs);
//   2-7    converters, three sets of two warps, set j filling stage slot j
//          (two weight rows per thread: nibbles -> sc*q binary16 in the
//          128-byte-swizzled K-major layout; the min operand once per
//          super-block).  The proxy fence that publishes a converted stage
//          to the tensor cores costs about as much as the conversion, so the
//          three sets keep three stages in flight;
//   8-15   epilogue (TMEM lane quarter = warp % 4, 128 token columns each),
//          holding the fp32 accumulator in registers: warpgroups 0-1 give
//          registers to warpgroups 2-3 (56 / 200 of the 128 per thread the
//          block is launched with).
// Every wait is bounded; a failed wait stops both CTAs of the pair.
#include <cuda.h>

#include "zq_cluster.cuh"
#include "zq_internal.cuh"
#include "zq_tc.cuh"
#include "zq_tc_common.cuh"

namespace zq {
namespace {

constexpr int kRows = 128;                 // weight rows per CTA (MMA M / 2)
constexpr int kToks = 128;                 // tokens staged per CTA (MMA N / 2)
constexpr int kPairM = 2 * kRows, kPairN = 2 * kToks;
constexpr int kStages = 3;                 // operand stages of K = 64
constexpr int kAtom = 128 * 128;           // 128 rows x 64 binary16 (128 B), 128-byte swizzle
constexpr int kMinAtom = 128 * 32;         // 128 rows x 16 binary16 (32 B), 32-byte swizzle
constexpr int kStageBytes = 3 * kAtom + 2 * kMinAtom;   // A (weights), B hi, B lo, A' (mins), B' (s8)
constexpr int kRawBytes = kRows * kQ4KBlockBytes;       // 128 rows x 144 B
constexpr int kThreads = 512;
constexpr int kConvWarp0 = 2, kConvWarps = 6;   // three sets of two warps, one set per stage slot
constexpr int kSetWarps = kConvWarps / kStages;
constexpr int kRawSlots = 3;               // raw Q4_K tiles, two super-blocks ahead
constexpr int kEpiWarp0 = 8, kEpiWarps = 8;
constexpr int kEpiCols = kPairN / 2;       // token columns per epilogue thread
constexpr uint32_t kIdesc = idesc_f16_f32(kPairM, kPairN);
constexpr uint32_t kTmemCols = 512;        // two accumulators of 256 columns
constexpr uint32_t kStageTx = 2 * 2 * kAtom;            // both CTAs' hi and lo token tiles
constexpr uint32_t kStageTxMin = kStageTx + 2 * kMinAtom;
constexpr uint32_t kSigTx = 4 * kSetWarps;                 // the odd CTA's converter signals
static_assert(kSetWarps * 32 * 2 == kRows, "a converter thread converts two weight rows of its stage");
static_assert(kEpiWarp0 % 4 == 0 && kEpiWarps == 8, "epilogue lane quarters follow warp % 4");

struct Smem {
    static constexpr size_t stage(int s) { return (size_t)s * kStageBytes; }
    static constexpr size_t a(int s) { return stage(s); }
    static constexpr size_t bhi(int s) { return stage(s) + kAtom; }
    static constexpr size_t blo(int s) { return stage(s) + 2 * kAtom; }
    static constexpr size_t amin(int s) { return stage(s) + 3 * kAtom; }
    static constexpr size_t bmin(int s) { return stage(s) + 3 * kAtom + kMinAtom; }
    static constexpr size_t raw(int i) { return stage(kStages) + (size_t)i * kRawBytes; }
    // words the odd CTA's converter warps store into (st.async) to signal a stage
    static constexpr size_t sig() { return raw(kRawSlots); }
    static constexpr size_t bars() { return sig() + 64; }
    // full[3], empty[3], raw_full[3], raw_empty[3], tfull[2], tempty[2], drain
    static constexpr int kNumBars = 2 * kStages + 2 * kRawSlots + 2 * 2 + 1;
    static constexpr size_t tmem_slot() { return bars() + kNumBars * 8; }
    static constexpr size_t total() { return tmem_slot() + 16 + 1024; }   // + alignment slack
};
static_assert(kStageBytes % 1024 == 0 && kRawBytes % 16 == 0, "operand atoms stay 1024-byte aligned");
static_assert(Smem::total() <= 227 * 1024, "shared memory budget");
static_assert(Smem::total() < (1u << 18), "descriptor start addresses stay inside their 14-bit field");

struct Pair2Params {
    int N, K, B, nb;
    int t_tiles;           // token tiles of 256
    int splits;            // K ranges; pair = (split, token tile, weight tile)
    size_t split_stride;   // floats between two splits' partial sums
    size_t row_bytes;      // bytes of one weight row (K/256 * 144)
    const uint8_t *W;
    const float *tscale;   // [B] power of two that undoes the code scaling
    float *y;              // [B][N], or [splits][split_stride] partial sums
    unsigned int *status;
};

// Per weight row and super-block: the factor applied to w = sc*q (a power of
// two, or 0 when d = 0), the ratio r whose binary16 parts carry the min term
// (-r * m_j), and the fold factor of the accumulator, so that
// fold * (wmul * w * x' - r * m * s8) = d * w * x' - dmin * m * s8.
struct Fold {
    float wmul, r, fold;
};

__device__ __forceinline__ Fold fold_params(uint32_t d_dmin)
{
    const float d = __half2float(__ushort_as_half((unsigned short)(d_dmin & 0xFFFFu)));
    const float dm = __half2float(__ushort_as_half((unsigned short)(d_dmin >> 16)));
    Fold f;
    float r = d != 0.0f ? dm / d : dm;
    const float base = d != 0.0f ? d : 1.0f;
    int e = 0;
    const float big = fabsf(r) * (63.0f / 16384.0f);   // |r * m| <= 16384 keeps the parts in binary16
    if (big > 1.0f) frexpf(big, &e);                     // big <= 2^e
    f.r = ldexpf(r, -e);
    f.wmul = d != 0.0f ? ldexpf(1.0f, -e) : 0.0f;
    f.fold = ldexpf(base, e);
    return f;
}

// Bounded wait on a barrier that may receive arrivals from the peer CTA;
// gives up at once when either CTA of the pair has already failed.  Inline
// throughout: a call out of a warpgroup whose register count was changed
// would force spills around it.
struct PairCtx {
    volatile int *abort_local;
    uint32_t abort_peer;   // cluster address of the peer's flag
    unsigned int *status;
};

__device__ __forceinline__ bool pair_wait(uint64_t *bar, uint32_t parity, const PairCtx &c)
{
    if (mbar_try_wait_cl(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (;;) {
        if (*c.abort_local) return false;
        if (mbar_try_wait_cl_sleep(bar, parity, kSleepNs)) return true;
        if (global_ns() - t0 >= kWaitLimitNs) {
            flag_timeout(c.status);
            *c.abort_local = 1;
            st_cluster_u32(c.abort_peer, 1u);
            return false;
        }
    }
}

__device__ __forceinline__ bool pair_warp_wait(uint64_t *bar, uint32_t parity, const PairCtx &c)
{
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = pair_wait(bar, parity, c);
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    if (ok) ok = pair_wait(bar, parity, c);
    return __all_sync(0xffffffffu, ok);
}

// Bounded wait that ignores the abort flags (draining work already issued).
__device__ __forceinline__ bool drain_wait(uint64_t *bar, uint32_t parity)
{
    const uint64_t t0 = global_ns();
    for (;;) {
        if (mbar_try_wait_cl_sleep(bar, parity, kSleepNs)) return true;
        if (global_ns() - t0 >= kWaitLimitNs) return false;
    }
}

// The pair's tile and K range, recomputed inside each role (after its
// register count changes) rather than kept live across the change.
struct Tile {
    int split, t0, m0, row0, b_begin, nb, rot;
    __device__ __forceinline__ int sb(int b) const { return b_begin + (b + rot < nb ? b + rot : b + rot - nb); }
};

__device__ __forceinline__ Tile tile_of(const Pair2Params &p, uint32_t rank)
{
    Tile t;
    const int pair = blockIdx.x >> 1;
    t.split = pair % p.splits;
    const int tile = pair / p.splits;
    const int t_tile = tile % p.t_tiles;
    const int m_tile = tile / p.t_tiles;
    t.t0 = t_tile * kPairN;
    t.m0 = m_tile * kPairM;
    t.row0 = t.m0 + kRows * (int)rank;
    t.b_begin = (int)((long long)t.split * p.nb / p.splits);
    t.nb = (int)((long long)(t.split + 1) * p.nb / p.splits) - t.b_begin;
    // both CTAs of a pair walk the same rotated super-block order; pairs with
    // different tiles start at different super-blocks
    t.rot = (m_tile + 5 * t_tile) % t.nb;
    return t;
}

__device__ __forceinline__ PairCtx pair_ctx(volatile int *abort_s, uint32_t rank, unsigned int *status)
{
    PairCtx c;
    c.abort_local = abort_s;
    c.abort_peer = cluster_addr(smem_u32(const_cast<int *>(abort_s)), rank ^ 1u);
    c.status = status;
    return c;
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

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
q4k_gemm_2sm_kernel(const __grid_constant__ CUtensorMap tmap_hi, const __grid_constant__ CUtensorMap tmap_lo,
                    const __grid_constant__ CUtensorMap tmap_s8, const __grid_constant__ CUtensorMap tmap_w,
                    const Pair2Params p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    __shared__ volatile int abort_s;

    uint64_t *bm = reinterpret_cast<uint64_t *>(sm + Smem::bars());
    uint64_t *full = bm, *empty = bm + kStages;
    uint64_t *raw_full = empty + kStages, *raw_empty = raw_full + kRawSlots;
    uint64_t *tfull = raw_empty + kRawSlots, *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + Smem::tmem_slot());

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            // the even CTA's producer and the slot's converter warps; the odd
            // CTA's converter warps signal with st.async bytes
            mbar_init(&full[s], 1 + kSetWarps);
            mbar_init(&empty[s], 1);
        }
        for (int i = 0; i < kRawSlots; ++i) {
            mbar_init(&raw_full[i], 1);
            mbar_init(&raw_empty[i], kConvWarps);   // every set converts part of every super-block
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], 2 * kEpiWarps);
        }
        mbar_init(drain, 1);
        abort_s = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc_pair(tmem_slot, kTmemCols);
    tc_fence_before();
    cluster_sync();   // barriers of both CTAs initialised, tensor memory allocated in both
    tc_fence_after();

    if (warp < kEpiWarp0) {
        regs_dec<56>();
        const uint32_t rank = cluster_rank();
        const Tile T = tile_of(p, rank);
        const PairCtx ctx = pair_ctx(&abort_s, rank, p.status);
        const int nb = T.nb;
        if (warp == 0) {
            // ------------------------------------------------ TMA producer
            if (lane == 0) {
                prefetch_tmap(&tmap_hi);
                prefetch_tmap(&tmap_lo);
                prefetch_tmap(&tmap_s8);
                prefetch_tmap(&tmap_w);
                const bool leader = rank == 0;
                const int tok0 = T.t0 + kToks * (int)rank;
                bool ok = true;
                auto load_raw = [&](int bb) -> bool {
                    const int slot = bb % kRawSlots, use = bb / kRawSlots;
                    if (use > 0 && !pair_wait(&raw_empty[slot], (use - 1) & 1, ctx)) return false;
                    mbar_arrive_expect_tx(&raw_full[slot], kRawBytes);
                    tma_load_2d(sm + Smem::raw(slot), &tmap_w, kQ4KBlockBytes * T.sb(bb), T.row0, &raw_full[slot]);
                    return true;
                };
                for (int bb = 0; bb < kRawSlots - 1 && bb < nb && ok; ++bb) ok = load_raw(bb);
                const int nq = 4 * nb;
                for (int q = 0; q < nq && ok; ++q) {
                    const int b = q >> 2, i = q & 3;
                    if (i == 0 && b + kRawSlots - 1 < nb && !(ok = load_raw(b + kRawSlots - 1))) break;
                    const int s = q % kStages, round = q / kStages;
                    if (round > 0 && !(ok = pair_wait(&empty[s], (round - 1) & 1, ctx))) break;
                    const uint32_t fb = cluster_addr(smem_u32(&full[s]), 0);
                    if (leader) mbar_arrive_expect_tx(&full[s], (i == 3 ? kStageTxMin : kStageTx) + kSigTx);
                    const int kx = 256 * T.sb(b) + 64 * i;
                    tma_load_2d_pair(sm + Smem::bhi(s), &tmap_hi, kx, tok0, fb);
                    tma_load_2d_pair(sm + Smem::blo(s), &tmap_lo, kx, tok0, fb);
                    if (i == 3) tma_load_2d_pair(sm + Smem::bmin(s), &tmap_s8, 16 * T.sb(b), tok0, fb);
                }
            }
        } else if (warp == 1) {
            // ------------------------------------------------ MMA issuer
            if (rank == 0 && lane == 0) {
                const uint32_t tmem = *tmem_slot;
                const uint32_t base = smem_u32(sm);
                const uint64_t a0 = smem_desc(base + (uint32_t)Smem::a(0), 16, 1024, kLayoutSw128);
                const uint64_t bh0 = smem_desc(base + (uint32_t)Smem::bhi(0), 16, 1024, kLayoutSw128);
                const uint64_t bl0 = smem_desc(base + (uint32_t)Smem::blo(0), 16, 1024, kLayoutSw128);
                const uint64_t am0 = smem_desc(base + (uint32_t)Smem::amin(0), 16, 256, kLayoutSw32);
                const uint64_t bm0 = smem_desc(base + (uint32_t)Smem::bmin(0), 16, 256, kLayoutSw32);
                constexpr uint64_t kStage16 = kStageBytes >> 4;
                int s = 0;
                uint32_t ph = 0;
                bool ok = true;
                for (int b = 0; b < nb && ok; ++b) {
                    const int buf = b & 1;
                    const uint32_t use = (uint32_t)(b >> 1);
                    const uint32_t d_tmem = tmem + (uint32_t)(kPairN * buf);
                    if (use > 0 && !(ok = pair_wait(&tempty[buf], (use - 1) & 1, ctx))) break;
                    tc_fence_after();
                    for (int i = 0; i < 4; ++i) {
                        if (!(ok = pair_wait(&full[s], ph, ctx))) break;
                        tc_fence_after();
                        const uint64_t so = (uint64_t)s * kStage16;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            mma_f16_pair(d_tmem, a0 + so + 2 * kk, bh0 + so + 2 * kk, kIdesc, (i | kk) != 0 ? 1u : 0u);
                            mma_f16_pair(d_tmem, a0 + so + 2 * kk, bl0 + so + 2 * kk, kIdesc, 1u);
                        }
                        if (i == 3) mma_f16_pair(d_tmem, am0 + so, bm0 + so, kIdesc, 1u);
                        mma_commit_pair_mc(&empty[s], 3);
                        if (++s == kStages) {
                            s = 0;
                            ph ^= 1u;
                        }
                    }
                    if (!ok) break;
                    mma_commit_pair_mc(&tfull[buf], 3);
                }
                // every MMA issued has completed before the pair tears down
                mma_commit_pair_local(drain);
                drain_wait(drain, 0);
            }
        } else if (warp >= kConvWarp0) {
            // ------------------------------------------------ converters
            // set j fills stage slot j (stages q = j, j + 3, ...); so three
            // stages are converted, fenced and published at once
            const int set = (warp - kConvWarp0) / kSetWarps;
            const int ct = ((warp - kConvWarp0) % kSetWarps) * 32 + lane;   // rows ct and ct + 64
            int cur_b = -1;
            bool ok = true;
            for (int q = set; q < 4 * nb && ok; q += kStages) {
                const int b = q >> 2, i = q & 3, round = q / kStages;
                if (b != cur_b) {
                    if (cur_b >= 0) {
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&raw_empty[cur_b % kRawSlots]);
                    }
                    if (!(ok = pair_warp_wait(&raw_full[b % kRawSlots], (uint32_t)(b / kRawSlots) & 1, ctx))) break;
                    cur_b = b;
                }
                if (round > 0 && !(ok = pair_warp_wait(&empty[set], (round - 1) & 1, ctx))) break;
#pragma unroll 1
                for (int h = 0; h < 2; ++h) {
                    const int r = ct + 64 * h;   // weight row within this CTA
                    const int sw = r & 7, s32 = (r >> 2) & 1;
                    const uint8_t *raw = sm + Smem::raw(b % kRawSlots) + (size_t)r * kQ4KBlockBytes;
                    const uint4 hdr = *reinterpret_cast<const uint4 *>(raw);
                    const Fold fp = fold_params(hdr.x);
                    const uint4 n0 = *reinterpret_cast<const uint4 *>(raw + 16 + 32 * i);
                    const uint4 n1 = *reinterpret_cast<const uint4 *>(raw + 32 + 32 * i);
                    uint32_t sc0, sc1, md;
                    q4k_scale_min(hdr.y, hdr.z, hdr.w, 2 * i, sc0, md);
                    q4k_scale_min(hdr.y, hdr.z, hdr.w, 2 * i + 1, sc1, md);
                    const float scl = (float)sc0 * fp.wmul, sch = (float)sc1 * fp.wmul;
                    const __half2 s_lo = __float2half2_rn(scl), o_lo = __float2half2_rn(-1024.0f * scl);
                    const __half2 s_hi = __float2half2_rn(sch * 0.0625f), o_hi = __float2half2_rn(-64.0f * sch);
                    const uint32_t wv[8] = {n0.x, n0.y, n0.z, n0.w, n1.x, n1.y, n1.z, n1.w};
                    uint8_t *arow = sm + Smem::a(set) + (size_t)r * 128;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint4 lo, hi;
                        nib4_to_h2<false>(wv[2 * c], s_lo, o_lo, lo.x, lo.y);
                        nib4_to_h2<false>(wv[2 * c + 1], s_lo, o_lo, lo.z, lo.w);
                        nib4_to_h2<true>(wv[2 * c], s_hi, o_hi, hi.x, hi.y);
                        nib4_to_h2<true>(wv[2 * c + 1], s_hi, o_hi, hi.z, hi.w);
                        *reinterpret_cast<uint4 *>(arow + ((c ^ sw) << 4)) = lo;
                        *reinterpret_cast<uint4 *>(arow + (((c + 4) ^ sw) << 4)) = hi;
                    }
                    if (i == 3) {
                        // the min operand: -r * m_j as binary16 hi (columns
                        // 0..7) and lo (8..15)
                        uint32_t hv[4], lv[4];
#pragma unroll
                        for (int j = 0; j < 8; j += 2) {
                            uint32_t m0v, m1v, scd;
                            q4k_scale_min(hdr.y, hdr.z, hdr.w, j, scd, m0v);
                            q4k_scale_min(hdr.y, hdr.z, hdr.w, j + 1, scd, m1v);
                            const float v0 = -fp.r * (float)m0v, v1 = -fp.r * (float)m1v;
                            const __half2 hh = __floats2half2_rn(v0, v1);
                            const float2 hb = __half22float2(hh);
                            hv[j >> 1] = h2_bits(hh);
                            lv[j >> 1] = h2_bits(__floats2half2_rn(v0 - hb.x, v1 - hb.y));
                        }
                        uint8_t *mrow = sm + Smem::amin(set) + (size_t)r * 32;
                        *reinterpret_cast<uint4 *>(mrow + ((0 ^ s32) << 4)) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
                        *reinterpret_cast<uint4 *>(mrow + ((1 ^ s32) << 4)) = make_uint4(lv[0], lv[1], lv[2], lv[3]);
                    }
                }
                fence_async_smem();
                __syncwarp();
                if (lane == 0) {
                    if (rank == 0)
                        mbar_arrive(&full[set]);
                    else
                        st_async_signal(cluster_addr(smem_u32(sm + Smem::sig()) + 4u * (warp - kConvWarp0), 0),
                                        cluster_addr(smem_u32(&full[set]), 0));
                }
            }
            if (ok && cur_b >= 0) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&raw_empty[cur_b % kRawSlots]);
            }
        }
    } else {
        regs_inc<200>();
        // ---------------------------------------------------- epilogue
        const uint32_t rank = cluster_rank();
        const Tile T = tile_of(p, rank);
        const PairCtx ctx = pair_ctx(&abort_s, rank, p.status);
        const int nb = T.nb;
        const uint32_t tmem = *tmem_slot;
        const int e = warp - kEpiWarp0;
        const int quarter = warp & 3;              // TMEM lanes 32*quarter .. +31
        const int half = e >> 2;                   // token columns 128*half ..
        const int n = T.row0 + 32 * quarter + lane;  // weight row
        const bool nvalid = n < p.N;
        const uint8_t *wrow = p.W + (size_t)(nvalid ? n : 0) * p.row_bytes;
        const uint32_t lane_base = tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(kEpiCols * half);
        const uint32_t tempty_leader0 = cluster_addr(smem_u32(&tempty[0]), 0);
        const uint32_t tempty_leader1 = cluster_addr(smem_u32(&tempty[1]), 0);
        float acc[kEpiCols];
#pragma unroll
        for (int c = 0; c < kEpiCols; ++c) acc[c] = 0.0f;
        uint32_t hd_next = nvalid ? ld_nc_u32(wrow + (size_t)kQ4KBlockBytes * T.sb(0)) : 0u;
        bool ok = true;
        for (int b = 0; b < nb && ok; ++b) {
            const int buf = b & 1;
            const uint32_t hd = hd_next;
            if (nvalid && b + 1 < nb) hd_next = ld_nc_u32(wrow + (size_t)kQ4KBlockBytes * T.sb(b + 1));
            const float fold = nvalid ? fold_params(hd).fold : 0.0f;
            if (!(ok = pair_warp_wait(&tfull[buf], (uint32_t)(b >> 1) & 1, ctx))) break;
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < kEpiCols / 16; ++c) {
                uint32_t v[16];
                tmem_ld16(lane_base + (uint32_t)(kPairN * buf) + 16u * c, v);
                tmem_wait_ld();
                if (c == kEpiCols / 16 - 1) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(buf ? tempty_leader1 : tempty_leader0);
                }
#pragma unroll
                for (int j = 0; j < 16; j += 2)
                    fma2(acc[16 * c + j], acc[16 * c + j + 1], fold, __uint_as_float(v[j]), __uint_as_float(v[j + 1]));
            }
        }
        if (ok && !abort_s && nvalid) {
            float *ybase = p.y + (size_t)T.split * p.split_stride + n;
            const int tc0 = T.t0 + kEpiCols * half;
#pragma unroll
            for (int c = 0; c < kEpiCols; ++c) {
                const int tok = tc0 + c;
                if (tok < p.B) ybase[(size_t)tok * p.N] = acc[c] * __ldg(p.tscale + tok);
            }
        }
    }
    __syncwarp();
    if (abort_s) {
        // a role gave up: let copies and signals already issued land before
        // the pair's shared memory goes away
        const uint64_t tw = global_ns();
        while (global_ns() - tw < 200000ull) {
        }
    }
    // back to the launch's 128 registers per thread before the roles meet
    // again (the epilogue's release lets the other warpgroups' request go on)
    if (warp < kEpiWarp0)
        regs_inc<128>();
    else
        regs_dec<128>();
    tc_fence_before();
    cluster_sync();   // the peer's MMAs, copies and arrivals are finished
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(*tmem_slot, kTmemCols);
    }
}

size_t g_attr_bytes[64];

}  // namespace

// Split-K count for 256 x 256 pair tiles on sms / 2 SM pairs: tiles that fill
// the pairs unevenly waste whole waves; model the time of `s` splits as
// waves * (super-blocks per split + a fixed cost) plus the partial-sum
// traffic, and take the smallest s within 3 % of the best (>= 2 super-blocks
// per split, s <= 8).
int choose_splits_pair(int B, int N, int K, int sms)
{
    const long long tiles = (long long)((B + kPairN - 1) / kPairN) * ((N + kPairM - 1) / kPairM);
    const int pairs = sms / 2 > 0 ? sms / 2 : 1;
    const int nb = K / 256;
    const int smax = nb / 2 < 8 ? nb / 2 : 8;
    double cost[9];
    double best = 1e300;
    for (int sp = 1; sp <= (smax > 1 ? smax : 1); ++sp) {
        const long long units = tiles * sp;
        const double waves = (double)((units + pairs - 1) / pairs);
        double c = waves * ((double)nb / sp + 1.0);
        if (sp > 1) c += (double)(sp + 1) * B * N * 4.0 / 1.5e7;   // partials, in super-block times
        cost[sp] = c;
        if (c < best) best = c;
    }
    for (int sp = 1; sp <= (smax > 1 ? smax : 1); ++sp)
        if (cost[sp] <= best * 1.03) return sp;
    return 1;
}

cudaError_t launch_gemm_pair(const void *W, int N, int K, int B, const __half *hi, const __half *lo,
                             const __half *s8x, const float *tscale, float *out, float *y, int splits, cudaStream_t st)
{
    CUtensorMap th, tl, ts, tw;
    const CUtensorMapDataType f16 = CU_TENSOR_MAP_DATA_TYPE_FLOAT16, u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
    cudaError_t e;
    if ((e = make_tmap_2d(&th, f16, 2, hi, (uint64_t)K, (uint64_t)B, 64, kToks, CU_TENSOR_MAP_SWIZZLE_128B)) !=
        cudaSuccess)
        return e;
    if ((e = make_tmap_2d(&tl, f16, 2, lo, (uint64_t)K, (uint64_t)B, 64, kToks, CU_TENSOR_MAP_SWIZZLE_128B)) !=
        cudaSuccess)
        return e;
    if ((e = make_tmap_2d(&ts, f16, 2, s8x, (uint64_t)K / 16, (uint64_t)B, 16, kToks, CU_TENSOR_MAP_SWIZZLE_32B)) !=
        cudaSuccess)
        return e;
    // weights as bytes [N][K/256*144]: one box = one super-block of 128 rows
    if ((e = make_tmap_2d(&tw, u8, 1, W, (uint64_t)(K / 256) * kQ4KBlockBytes, (uint64_t)N, kQ4KBlockBytes, kRows,
                          CU_TENSOR_MAP_SWIZZLE_NONE)) != cudaSuccess)
        return e;
    Pair2Params p{};
    p.N = N;
    p.K = K;
    p.B = B;
    p.nb = K / 256;
    p.t_tiles = (B + kPairN - 1) / kPairN;
    p.splits = splits;
    p.split_stride = split_stride(B, N);
    p.row_bytes = (size_t)(K / 256) * kQ4KBlockBytes;
    p.W = static_cast<const uint8_t *>(W);
    p.tscale = tscale;
    p.y = out;
    p.status = device_status_word();
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    const size_t smem = Smem::total();
    if (g_attr_bytes[dev] < smem) {
        e = cudaFuncSetAttribute(q4k_gemm_2sm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        g_attr_bytes[dev] = smem;
    }
    const long long pairs = (long long)p.t_tiles * ((N + kPairM - 1) / kPairM) * splits;
    q4k_gemm_2sm_kernel<<<(unsigned)(2 * pairs), kThreads, smem, st>>>(th, tl, ts, tw, p);
    if (splits == 1) return cudaGetLastError();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    return launch_splitk_reduce(out, splits, (size_t)B * N, y, st);
}

}  // namespace zq
