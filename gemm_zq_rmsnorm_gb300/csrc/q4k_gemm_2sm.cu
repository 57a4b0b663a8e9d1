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
// Tile of a CTA pair: 256 weight rows (the MMA's M: 128 rows in each CTA) x
// 256 tokens (the MMA's N: each CTA stages 128 tokens, the MMA reads both
// halves).  Each CTA converts only its own 128 weight rows, and every
// converted weight meets all 256 tokens; one 256 x 256 x 16 MMA keeps each
// SM's tensor core busy for ~128 cycles.
//
// The converted weights (the MMA's A operand) go to tensor memory with
// tcgen05.st, not to shared memory: shared memory then carries only the
// token tiles (TMA writes, MMA reads), the raw Q4_K tiles and the small min
// operands, and the MMA's reads of A no longer compete with the converters
// for its bandwidth (with A in shared memory the converters were starved).
// Tensor memory (512 columns): the accumulator (256 columns, tokens) and
// eight A slots of 32 columns (a K = 64 stage of binary16 weights, two
// super-blocks ahead).  The accumulator is single-buffered: the MMAs of
// super-block b+1 wait for the epilogue to read X_b (~600 cycles per
// super-block of ~4200 MMA cycles).
//
// Stage q (a quarter of a super-block, K = 64) has one "full" barrier in the
// even CTA, in A slot q % 8: the token tiles' TMA bytes of both CTAs and the
// converter warps of both CTAs complete it, so the MMA issuer waits once per
// stage.  One commit per stage ("empty") frees A slot q % 8 and the token
// slot of stage q (MMAs complete in order, so the producer waits on the
// barrier of the stage that last used its slot).
//
// Warp roles (16 warps, four warpgroups):
//   0      token TMA producer: the binary16 hi/lo token tiles (five stages)
//          and the s8 tiles, whose bytes are counted on the even CTA's stage
//          barrier;
//   1      MMA issuer (even CTA only) and tensor-memory owner (both CTAs);
//   2      raw-tile TMA producer: the Q4_K tiles of this CTA's 128 rows (two
//          super-block slots);
//   3      idle;
//   4-7    converters, one weight row per thread (TMEM lane = row): nibbles
//          -> sc*q binary16 in registers -> tensor memory; the odd CTA's
//          warps signal a converted stage to the even CTA's barrier with
//          st.async (a cluster-scope release-arrive costs ~1200 cycles);
//   8-15   epilogue (TMEM lane quarter = warp % 4, 128 token columns each),
//          holding the fp32 accumulator in registers: warpgroups 0-1 give
//          registers to warpgroups 2-3 (64 / 192 of the 128 per thread the
//          block is launched with).  One lane polls the accumulator's
//          barrier without sleeping and releases the others through a
//          hardware named barrier.
// Every wait is bounded; a failed wait stops both CTAs of the pair.
#include <cuda.h>

#include "zq_cluster.cuh"
#include "zq_pair_wait.cuh"
#include "zq_internal.cuh"
#include "zq_tc.cuh"
#include "zq_tc_common.cuh"
#include "q4k_tc_convert.cuh"

namespace zq {
namespace {

constexpr int kRows = 128;                 // weight rows per CTA (MMA M / 2)
constexpr int kTileN = 256;                // tokens per pair tile (MMA N, at most)
constexpr int kToks = kTileN / 2;          // tokens staged per CTA
constexpr int kPairM = 2 * kRows;
constexpr int kStages = 5;                 // K = 64 token stages (a super-block is four)
constexpr int kASlots = 8;                 // K = 64 converted-weight stages in tensor memory
constexpr int kAtom = kToks * 128;         // 128 token rows x 64 binary16 (128 B), 128-byte swizzle
constexpr int kMinAtom = 128 * 32;         // 128 rows x 16 binary16 (32 B), 32-byte swizzle
constexpr int kBStageBytes = 2 * kAtom;    // hi, lo
constexpr int kRawSlots = 2;               // raw Q4_K tiles
constexpr int kRawBytes = kRows * kQ4KBlockBytes;       // 128 rows x 144 B
constexpr int kThreads = 512;
constexpr int kConvWarp0 = 4, kConvWarps = 4;
constexpr int kEpiWarp0 = 8, kEpiWarps = 8;
constexpr int kEpiCols = kTileN / 2;       // token columns per epilogue thread
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kACol0 = kTileN, kACols = 32;        // accumulator [0, 256), A slot k at 256 + 32 k
constexpr uint32_t kConvSigTx = 4 * kConvWarps;         // the odd CTA's converter signals
constexpr uint32_t kEpiSigTx = 4 * kEpiWarps;           // the odd CTA's epilogue signals
static_assert(kConvWarps * 32 == kRows && kConvWarp0 % 4 == 0, "one converter thread per row, warp % 4 = quarter");
static_assert(kEpiWarp0 % 4 == 0 && kEpiWarps == 8 && kEpiCols % 32 == 0, "epilogue lane quarters follow warp % 4");
static_assert(kACol0 + kASlots * kACols <= kTmemCols, "tensor memory budget");
static_assert(kToks % 8 == 0 && kTileN % 16 == 0, "MMA N and the swizzle atoms' 8-row groups");

struct Smem {
    static constexpr size_t bhi(int s) { return (size_t)s * kBStageBytes; }
    static constexpr size_t blo(int s) { return bhi(s) + kAtom; }
    static constexpr size_t bmin(int i) { return (size_t)kStages * kBStageBytes + (size_t)i * kMinAtom; }  // s8 tiles, 2 slots
    static constexpr size_t amin(int i) { return bmin(2) + (size_t)i * kMinAtom; }     // min operand, 2 slots
    static constexpr size_t raw(int i) { return amin(2) + (size_t)i * kRawBytes; }
    // words the odd CTA's warps store into (st.async) to signal the even CTA
    static constexpr size_t sig() { return raw(kRawSlots); }
    static constexpr size_t bars() { return sig() + 64; }
    // full[8], empty[8], raw_full[2], raw_empty[2], tfull, tempty, drain
    static constexpr int kNumBars = 2 * kASlots + 2 * kRawSlots + 3;
    static constexpr size_t tmem_slot() { return bars() + kNumBars * 8; }
    static constexpr size_t total() { return tmem_slot() + 16 + 1024; }   // + alignment slack
};
static_assert(kBStageBytes % 1024 == 0 && kRawBytes % 16 == 0, "operand atoms aligned");
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

// The pair's tile and K range, recomputed inside each role (after its
// register count changes) rather than kept live across the change.
struct Tile {
    int split, t0, n, m0, row0, b_begin, nb, rot;   // n: the tile's tokens (MMA N, a multiple of 16)
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
    t.t0 = t_tile * kTileN;
    t.n = min(kTileN, (p.B - t.t0 + 15) & ~15);
    t.m0 = m_tile * kPairM;
    t.row0 = t.m0 + kRows * (int)rank;
    t.b_begin = (int)((long long)t.split * p.nb / p.splits);
    t.nb = (int)((long long)(t.split + 1) * p.nb / p.splits) - t.b_begin;
    // both CTAs of a pair walk the same rotated super-block order; pairs with
    // different tiles start at different super-blocks
    t.rot = (m_tile + 5 * t_tile) % t.nb;
    return t;
}


__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
q4k_gemm_2sm_kernel(const __grid_constant__ CUtensorMap tmap_hi, const __grid_constant__ CUtensorMap tmap_lo,
                    const __grid_constant__ CUtensorMap tmap_s8, const __grid_constant__ CUtensorMap tmap_w,
                    const Pair2Params p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);

    uint64_t *bm = reinterpret_cast<uint64_t *>(sm + Smem::bars());
    // full[k]: stage q (k = q % 8) is ready: its token tiles landed (TMA bytes
    // of both CTAs) and its weights are in tensor memory (both CTAs'
    // converters); empty[k]: the MMAs of stage q have completed, which frees
    // A slot k and the token slot of stage q (MMAs complete in order)
    uint64_t *afull = bm, *aempty = bm + kASlots;
    uint64_t *raw_full = aempty + kASlots, *raw_empty = raw_full + kRawSlots;
    uint64_t *tfull = raw_empty + kRawSlots, *tempty = tfull + 1, *drain = tempty + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + Smem::tmem_slot());

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int k = 0; k < kASlots; ++k) {
            // the even CTA's token producer and converter warps (+ the TMA
            // bytes of both CTAs and the odd CTA's st.async bytes)
            mbar_init(&afull[k], 1 + kConvWarps);
            mbar_init(&aempty[k], 1);
        }
        for (int i = 0; i < kRawSlots; ++i) {
            mbar_init(&raw_full[i], 1);
            mbar_init(&raw_empty[i], kConvWarps);
        }
        mbar_init(tfull, 1);
        mbar_init(tempty, kEpiWarps);   // the even CTA's epilogue warps (+ the odd CTA's st.async bytes)
        mbar_init(drain, 1);
        s_abort = 0;
        s_status = p.status;
        fence_mbar_init();
        pdl_launch_dependents();
    }
    if (warp == 1) tmem_alloc_pair(tmem_slot, kTmemCols);
    tc_fence_before();
    cluster_sync();   // barriers of both CTAs initialised, tensor memory allocated in both
    tc_fence_after();

    if (warp < kEpiWarp0) {
        regs_dec<64>();
        const uint32_t rank = cluster_rank();
        const Tile T = tile_of(p, rank);
        const PairCtx ctx = pair_ctx(rank);
        const int nb = T.nb;
        if (warp == 0) {
            if (lane == 0) {
                // ------------------------------------------ token tiles
                // CTA r stages the tile's tokens r*n/2 .. (96 rows; the MMA
                // reads the first n/2).  The tokens may come from the
                // previous kernel on the stream (programmatic launch): wait
                // for it first; the weights, set-up and conversion do not.
                pdl_wait();
                prefetch_tmap(&tmap_hi);
                prefetch_tmap(&tmap_lo);
                prefetch_tmap(&tmap_s8);
                const int tok0 = T.t0 + (T.n >> 1) * (int)rank;
                const uint32_t tx = 2u * (uint32_t)kBStageBytes, tx_min = tx + 2u * kToks * 32u;
                bool ok = true;
                for (int q = 0; q < 4 * nb && ok; ++q) {
                    const int b = q >> 2, i = q & 3;
                    const int s = q % kStages, k = q % kASlots;
                    // token slot s last held stage q - 5, whose MMAs completing
                    // arrive on empty[(q - 5) % 8]
                    if (q >= kStages &&
                        !(ok = pair_wait(&aempty[(q - kStages) % kASlots], ((q - kStages) / kASlots) & 1, ctx)))
                        break;
                    const uint32_t fb = cluster_addr(smem_u32(&afull[k]), 0);
                    if (rank == 0) mbar_arrive_expect_tx(&afull[k], i == 3 ? tx_min : tx);
                    const int kx = 256 * T.sb(b) + 64 * i;
                    tma_load_2d_pair(sm + Smem::bhi(s), &tmap_hi, kx, tok0, fb);
                    tma_load_2d_pair(sm + Smem::blo(s), &tmap_lo, kx, tok0, fb);
                    // the s8 tile of super-block b (slot b & 1): its previous
                    // reader, the min MMA of b - 2, finished before the MMAs
                    // of the stage this slot held last
                    if (i == 3) tma_load_2d_pair(sm + Smem::bmin(b & 1), &tmap_s8, 16 * T.sb(b), tok0, fb);
                }
            }
        } else if (warp == 2) {
            // (a warp of its own: a lane of the token producer's warp waiting
            // on the raw ring would hold that warp's token copies back)
            if (lane == 0) {
                // ------------------------------------------ raw Q4_K tiles
                prefetch_tmap(&tmap_w);
                for (int bb = 0; bb < nb; ++bb) {
                    const int slot = bb % kRawSlots, use = bb / kRawSlots;
                    if (use > 0 && !pair_wait(&raw_empty[slot], (use - 1) & 1, ctx)) break;
                    mbar_arrive_expect_tx(&raw_full[slot], kRawBytes);
                    tma_load_2d(sm + Smem::raw(slot), &tmap_w, kQ4KBlockBytes * T.sb(bb), T.row0, &raw_full[slot]);
                }
            }
        } else if (warp == 1) {
            // ------------------------------------------------ MMA issuer
            // (the whole warp runs the loop and waits; one elected lane issues)
            if (rank == 0) {
                const uint32_t tmem = *tmem_slot;
                const uint32_t base = smem_u32(sm);
                const uint64_t bh0 = smem_desc(base + (uint32_t)Smem::bhi(0), 16, 1024, kLayoutSw128);
                const uint64_t bl0 = smem_desc(base + (uint32_t)Smem::blo(0), 16, 1024, kLayoutSw128);
                const uint64_t bmn = smem_desc(base + (uint32_t)Smem::bmin(0), 16, 256, kLayoutSw32);
                const uint64_t am0 = smem_desc(base + (uint32_t)Smem::amin(0), 16, 256, kLayoutSw32);
                constexpr uint64_t kB16 = kBStageBytes >> 4, kM16 = kMinAtom >> 4;
                const uint32_t idesc = idesc_f16_f32(kPairM, (uint32_t)T.n);
                bool ok = true;
                for (int q = 0; q < 4 * nb && ok; ++q) {
                    const int b = q >> 2, i = q & 3;
                    const int k = q % kASlots;
                    if (i == 0 && b > 0) {
                        // the epilogue has read X_{b-1}
                        if (!(ok = __all_sync(0xffffffffu, pair_wait_spin(tempty, (b - 1) & 1, ctx)))) break;
                    }
                    const int s = q % kStages;
                    if (!(ok = __all_sync(0xffffffffu, pair_wait_spin(&afull[k], (q / kASlots) & 1, ctx)))) break;
                    tc_fence_after();
                    const uint32_t a_tmem = tmem + kACol0 + kACols * k;
                    const uint64_t so = (uint64_t)s * kB16;
                    if (elect_one()) {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            mma_f16_pair_ta(tmem, a_tmem + 8 * kk, bh0 + so + 2 * kk, idesc, (i | kk) != 0 ? 1u : 0u);
                            mma_f16_pair_ta(tmem, a_tmem + 8 * kk, bl0 + so + 2 * kk, idesc, 1u);
                        }
                        if (i == 3) {
                            mma_f16_pair(tmem, am0 + (uint64_t)(b & 1) * kM16, bmn + (uint64_t)(b & 1) * kM16, idesc,
                                         1u);
                            mma_commit_pair_mc(tfull, 3);
                        }
                        mma_commit_pair_mc(&aempty[k], 3);
                    }
                    __syncwarp();
                }
                // every MMA issued has completed before the pair tears down
                if (elect_one()) mma_commit_pair_local(drain);
                __syncwarp();
                drain_wait(drain, 0);
            }
        } else if (warp >= kConvWarp0) {
            // ------------------------------------------------ converters
            const uint32_t tmem = *tmem_slot;
            const int r = threadIdx.x - 32 * kConvWarp0;   // weight row = TMEM lane
            const uint32_t lane_base = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + kACol0;
            const uint32_t sig = cluster_addr(smem_u32(sm + Smem::sig()) + 4u * (warp - kConvWarp0), 0);
            const uint32_t afull_cl0 = cluster_addr(smem_u32(&afull[0]), 0);   // barriers 8 bytes apart
            int cur_b = -1;
            bool ok = true;
            for (int q = 0; q < 4 * nb && ok; ++q) {
                const int b = q >> 2, i = q & 3;
                const int k = q % kASlots, round = q / kASlots;
                if (b != cur_b) {
                    if (cur_b >= 0 && lane == 0) mbar_arrive(&raw_empty[cur_b % kRawSlots]);
                    if (!(ok = pair_warp_wait(&raw_full[b % kRawSlots], (uint32_t)(b / kRawSlots) & 1, ctx))) break;
                    cur_b = b;
                }
                if (round > 0 && !(ok = pair_warp_wait(&aempty[k], (round - 1) & 1, ctx))) break;
                tc_fence_after();
                const uint8_t *raw = sm + Smem::raw(b % kRawSlots) + (size_t)r * kQ4KBlockBytes;
                const uint32_t col = lane_base + kACols * k;
                uint8_t *mrow = sm + Smem::amin(b & 1) + (size_t)r * 32;
                switch (i) {
                case 0: convert_one<0>(raw, col, mrow, r); break;
                case 1: convert_one<1>(raw, col, mrow, r); break;
                case 2: convert_one<2>(raw, col, mrow, r); break;
                default: convert_one<3>(raw, col, mrow, r); break;
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (rank != 0)
                        st_async_signal(sig, afull_cl0 + 8u * (uint32_t)k);
                    else if (warp == kConvWarp0)
                        mbar_arrive_expect_tx(&afull[k], kConvSigTx);
                    else
                        mbar_arrive(&afull[k]);
                }
            }
            if (ok && cur_b >= 0) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&raw_empty[cur_b % kRawSlots]);
            }
        }
    } else {
        regs_inc<192>();
        // ---------------------------------------------------- epilogue
        // (y, the partial sums and the token scales belong to the stream's
        // previous kernels until they complete)
        pdl_wait();
        const uint32_t rank = cluster_rank();
        const Tile T = tile_of(p, rank);
        const PairCtx ctx = pair_ctx(rank);
        const int nb = T.nb;
        const uint32_t tmem = *tmem_slot;
        const int e = warp - kEpiWarp0;
        const int quarter = warp & 3;              // TMEM lanes 32*quarter .. +31
        const int half = e >> 2;                   // token columns 128*half ..
        const int n = T.row0 + 32 * quarter + lane;  // weight row
        const bool nvalid = n < p.N;
        const uint32_t lane_base = tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(kEpiCols * half);
        const uint32_t sig = cluster_addr(smem_u32(sm + Smem::sig()) + 16u + 4u * e, 0);
        const uint32_t tempty_cl = cluster_addr(smem_u32(tempty), 0);
        float acc[kEpiCols];
#pragma unroll
        for (int c = 0; c < kEpiCols; ++c) acc[c] = 0.0f;
        uint32_t hd_next = nvalid ? ld_nc_u32(p.W + (size_t)n * p.row_bytes + (size_t)kQ4KBlockBytes * T.sb(0)) : 0u;
        bool ok = true;
        for (int b = 0; b < nb && ok; ++b) {
            const uint32_t hd = hd_next;
            if (nvalid && b + 1 < nb)
                hd_next = ld_nc_u32(p.W + (size_t)n * p.row_bytes + (size_t)kQ4KBlockBytes * T.sb(b + 1));
            const float fold = nvalid ? fold_of(hd).fold : 0.0f;
            // one lane polls without sleeping; the others wait at a hardware
            // barrier, which wakes them within a few cycles
            if (e == 0) ok = pair_lane0_wait_spin(tfull, (uint32_t)b & 1, ctx);
            named_bar(1, 32 * kEpiWarps);
            if (!(ok = !*reinterpret_cast<volatile int *>(&s_abort))) break;
            tc_fence_after();
#pragma unroll
            for (int h = 0; h < kEpiCols / 32; ++h) {
                uint32_t v[32];
                tmem_ld16(lane_base + 32u * h, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
                tmem_ld16(lane_base + 32u * h + 16u, *reinterpret_cast<uint32_t(*)[16]>(&v[16]));
                tmem_wait_ld();
                if (h == kEpiCols / 32 - 1) {
                    // X_b is read: the MMAs of super-block b + 1 may overwrite it
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        if (rank != 0)
                            st_async_signal(sig, tempty_cl);
                        else if (e == 0)
                            mbar_arrive_expect_tx(tempty, kEpiSigTx);
                        else
                            mbar_arrive(tempty);
                    }
                }
#pragma unroll
                for (int j = 0; j < 32; j += 2)
                    fma2(acc[32 * h + j], acc[32 * h + j + 1], fold, __uint_as_float(v[j]), __uint_as_float(v[j + 1]));
            }
        }
        if (ok && !*reinterpret_cast<volatile int *>(&s_abort) && nvalid) {
            float *ybase = p.y + (size_t)T.split * p.split_stride + n;
            const int tc0 = T.t0 + kEpiCols * half;   // column c <-> token t0 + c
#pragma unroll
            for (int c = 0; c < kEpiCols; ++c) {
                const int tok = tc0 + c;
                if (tok < p.B && kEpiCols * half + c < T.n) ybase[(size_t)tok * p.N] = acc[c] * __ldg(p.tscale + tok);
            }
        }
    }
    __syncwarp();
    if (*reinterpret_cast<volatile int *>(&s_abort)) {
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
    cluster_sync();   // the peer's MMAs, copies and signals are finished
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(*tmem_slot, kTmemCols);
    }
}

size_t g_attr_bytes[64];

}  // namespace

// Split-K count for 256-row x 192-token pair tiles on sms / 2 SM pairs: tiles that fill
// the pairs unevenly waste whole waves; model the time of `s` splits as
// waves * (super-blocks per split + a fixed cost) plus the partial-sum
// traffic, and take the smallest s within 3 % of the best (>= 2 super-blocks
// per split, s <= 8).
int choose_splits_pair(int B, int N, int K, int sms)
{
    const long long tiles = (long long)((B + kTileN - 1) / kTileN) * ((N + kPairM - 1) / kPairM);
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
    p.t_tiles = (B + kTileN - 1) / kTileN;
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
    if ((e = launch_pdl(q4k_gemm_2sm_kernel, dim3((unsigned)(2 * pairs)), dim3(kThreads), smem, st, th, tl, ts, tw,
                        p)) != cudaSuccess)
        return e;
    if (splits == 1) return cudaSuccess;
    return launch_splitk_reduce(out, splits, (size_t)B * N, y, st);
}

}  // namespace zq
