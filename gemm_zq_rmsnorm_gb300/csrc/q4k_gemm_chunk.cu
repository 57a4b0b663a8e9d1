// q4k_gemm_chunk.cu -- Q4_K x Q8_1 projection of a chunk of tokens
// (2 <= B <= 16) on the tensor cores of CTA pairs.
//
// MIInfer README, "Current phase": token-batched chunk projections that read
// each weight once for the whole chunk (chunks of four to sixteen tokens).
//
// A chunk is bound by HBM: every weight is read once and serves only B <= 16
// tokens, so the kernel must turn Q4_K bytes into MMA operands as fast as
// HBM delivers them (~80 weights per ns per SM).  Measured on this GPU, a
// tcgen05 kind::f16 MMA of 128 rows x K = 16 takes ~20 ns per SM whatever
// N <= 32 when issued from a warp-wide loop (~37 ns from a one-lane loop), so
// each MMA must carry as many weights as possible and nothing else:
//   * A CTA pair runs 256 x 32 x 16 MMAs (cta_group::2): 128 weight rows per
//     SM (A, converted to binary16 sc*q in tensor memory by converter warps),
//     and N = 32 token columns: the binary16 hi halves of x' = q8*d8 of the
//     16 tokens (even CTA's shared memory) and their lo halves (odd CTA's),
//     so one MMA covers both halves and every product is exact.
//   * The min term of a super-block enters the same accumulator through one
//     more MMA (A = -(dmin/d)*m_j as binary16 hi and lo parts, B = the
//     tokens' scaled s8 values twice in the hi columns, zeros in the lo
//     columns): 17 MMAs per super-block of 256 rows x 256 weights.
//   * The epilogue folds acc[t] += fold_b * (X_hi[t] + X_lo[t]) per row and
//     super-block from a ring of four accumulators (32 columns each).
// Work: the (256-row tile, super-block) sequence of the matrix is cut into
// one contiguous range per CTA pair, so every pair streams the same number
// of weight bytes whatever the shape; a tile that straddles ranges leaves
// partial sums per range, which a fixup kernel adds in range order.
//
// Warp roles (28 warps): 0 the token loader (cp.async copies of each
// super-block's token tiles and s8 tile into an eight-super-block ring,
// signalled to the even CTA's barrier); 1 the MMA issuer (even CTA, whole
// warp, one elected lane: the 17 MMAs of a super-block back to back) and
// tensor-memory owner; 2 the raw-tile TMA producer (this CTA's Q4_K
// super-block tiles, six in flight); 3 idle; 4-19 converters, one per (TMEM
// lane quarter w % 4, K = 64 stage (w - 4) / 4): the stage's two sub-block
// scales come from shared memory, so a converter only turns nibbles into
// binary16 products; 20-23 one per lane quarter: they decode each row's
// super-block metadata once (sub-block scales, the min operand, the fold)
// into a ring of their own as soon as the raw tile lands, so the converters
// find it ready; 24-27 the epilogue, one per lane quarter.  The integer pipe bounds the converters:
// one byte permute per four weights, two masks per four and one half2 fused
// multiply-add per two; sixteen of them keep enough independent work in
// flight on each SM sub-partition.
// Waits suspend in hardware rather than spin, leaving issue slots to the
// converters, which share every SM sub-partition with the other roles (a
// warp reaches only the TMEM lane quarter of its sub-partition).  Every wait
// is bounded; a failed wait stops both CTAs of the pair.
#include <cuda.h>

#include "q4k_tc_convert.cuh"
#include "zq_cluster.cuh"
#include "zq_internal.cuh"
#include "zq_pair_wait.cuh"
#include "zq_tc.cuh"
#include "zq_tc_common.cuh"

namespace zq {
namespace {

constexpr int kRows = 128;                  // weight rows per CTA
constexpr int kPairM = 2 * kRows;
constexpr int kTok = 16;                    // tokens (hi columns 0..15, lo columns 16..31)
constexpr int kN = 2 * kTok;
constexpr int kASB = 3;                     // super-blocks of converted weights in TMEM (four K = 64 stages each)
constexpr int kAcc = 4;                     // super-block accumulators
constexpr int kRawSlots = 6;                // raw Q4_K tiles (110 KB in flight)
constexpr int kMetaSlots = 6;               // decoded row metadata (sub-block scales, min operand) ring
constexpr int kTokSB = 8;                   // token ring, in super-blocks (four K = 64 stages and an s8 tile each)
constexpr int kTokAtom = kTok * 128;        // 16 rows x 64 binary16, 128-byte swizzle
constexpr int kAMinAtom = kRows * 32;       // 128 rows x 16 binary16, 32-byte swizzle
constexpr int kBMinAtom = kTok * 32;        // 16 rows x 16 binary16, 32-byte swizzle
constexpr int kRawBytes = kRows * kQ4KBlockBytes;
constexpr int kThreads = 896;
constexpr int kConvWarp0 = 4, kConvWarps = 16;  // one per (TMEM lane quarter, K = 64 stage)
constexpr int kMetaWarp0 = 20, kMetaWarps = 4;  // row metadata, one per lane quarter
constexpr int kEpiWarp0 = 24, kEpiWarps = 4;    // epilogue, one per lane quarter
constexpr int kScaleRow = 16;                   // bytes per row of a super-block's sub-block scales
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kACol0 = kAcc * kN, kACols = 128;  // accumulators [0, 128), A slot a at 128 + 128 a
constexpr uint32_t kConvSigTx = 4 * kConvWarps;        // the odd CTA's converter warps
constexpr uint32_t kTokSigTx = 4;                      // the odd CTA's token relay (warp 1)
constexpr uint32_t kEpiSigTx = 4 * kEpiWarps;          // the odd CTA's epilogue warps
static_assert(kACol0 + kASB * kACols <= kTmemCols, "tensor memory budget");

struct Smem {
    // token slot ts holds the four stages of one super-block, then its s8 tile
    static constexpr size_t tok(int ts, int i) { return ((size_t)ts * 4 + i) * kTokAtom; }
    static constexpr size_t bmin(int ts) { return tok(kTokSB, 0) + (size_t)ts * kBMinAtom; }
    static constexpr size_t amin(int i) { return bmin(kTokSB) + (size_t)i * kAMinAtom; }
    // the eight sub-block scales sc_j * 2^-e of each row (binary16), per metadata slot
    static constexpr size_t scales(int i) { return amin(kMetaSlots) + (size_t)i * kRows * kScaleRow; }
    // each row's accumulator fold (fp32), per metadata slot
    static constexpr size_t fold(int i) { return scales(kMetaSlots) + (size_t)i * kRows * 4; }
    static constexpr size_t raw(int i) { return fold(kMetaSlots) + (size_t)i * kRawBytes; }
    static constexpr size_t sig() { return raw(kRawSlots); }   // st.async targets of the odd CTA's warps
    static constexpr size_t bars() { return sig() + 128; }
    // afull[3], aempty[3], raw_full[6], raw_empty[6], tfull[4], tempty[4],
    // tok_full[8], tok_empty[8], drain, meta_full[6], meta_empty[6], tok_land[8]
    static constexpr int kNumBars = 2 * kASB + 2 * kRawSlots + 2 * kAcc + 3 * kTokSB + 1 + 2 * kMetaSlots;
    static constexpr size_t tmem_slot() { return bars() + kNumBars * 8; }
    static constexpr size_t total() { return tmem_slot() + 16 + 1024; }   // + alignment slack
};
static_assert(Smem::bmin(0) % 1024 == 0 && Smem::amin(0) % 256 == 0 && Smem::raw(0) % 128 == 0, "atom alignment");
static_assert(kTokAtom % 1024 == 0, "token atoms stay 1024-byte aligned");
static_assert(Smem::total() <= 227 * 1024, "shared memory budget");
static_assert(Smem::total() < (1u << 18), "descriptor start addresses stay inside their 14-bit field");

struct ChunkParams {
    int N, K, B, nb;
    int tiles;             // 256-row tiles
    long long total;       // tiles * nb super-blocks
    size_t row_bytes;
    const uint8_t *W;
    const float *tscale;   // [B]
    const __half *hi, *lo; // [B][K] binary16 parts of the activations
    const __half *s8x;     // [B][K/16] scaled s8 values, twice per super-block
    float *y;              // [B][N]
    float *part;           // [pieces][B][N] partial sums of straddling tiles
    unsigned int *status;
};

// Contiguous ranges: pair p takes the global super-blocks [r(p), r(p+1)) of
// the sequence tile * nb + b; the pair holding super-block g is the largest p
// with r(p) <= g.
__host__ __device__ inline long long range_start(int p, long long total, int P)
{
    return (long long)p * total / P;
}

__host__ __device__ inline int pair_of(long long g, long long total, int P)
{
    int p = (int)(g * P / total);
    while (p + 1 < P && range_start(p + 1, total, P) <= g) ++p;
    while (p > 0 && range_start(p, total, P) > g) --p;
    return p;
}

__device__ __forceinline__ void signal_leader(uint64_t *bar_local, uint32_t rank, bool expect, uint32_t tx,
                                              uint32_t sig_cl, uint32_t bar_cl)
{
    if (rank != 0)
        st_async_signal(sig_cl, bar_cl);
    else if (expect)
        mbar_arrive_expect_tx(bar_local, tx);
    else
        mbar_arrive(bar_local);
}

// 2^-e of a weight row's super-block (0 when d = 0): e from the binary16
// exponents of d and dmin alone, as in fold_of.
__device__ __forceinline__ float weight_scale(uint32_t d_dmin, int &e)
{
    const uint32_t hd = d_dmin & 0x7FFFu, hm = (d_dmin >> 16) & 0x7FFFu;
    e = hm ? max(0, f16_ilog2(hm) - (hd ? f16_ilog2(hd) : 0) - 7) : 0;
    return hd ? __int_as_float((127 - e) << 23) : 0.0f;
}

// Decodes the super-block metadata of one weight row: the eight sub-block
// scales sc_j * 2^-e as binary16 into `srow` (s_j at half j), the min
// operand -(dmin/d) * m_j * 2^-e as binary16 hi and lo parts into the row's
// 32-byte swizzled line `mrow` (hi parts in its first 16 bytes, lo parts in
// the second, before the swizzle), and returns the accumulator's fold
// (d, or 1 when d = 0) * 2^e.
__device__ __forceinline__ float decode_row(const uint8_t *raw, uint8_t *srow, uint8_t *mrow, int r)
{
    const uint4 hdr = *reinterpret_cast<const uint4 *>(raw);
    int e;
    const float wmul = weight_scale(hdr.x, e);
    // min terms: r = dmin / d (dmin itself when d = 0), times 2^-e
    const float d = __half2float(__ushort_as_half((unsigned short)(hdr.x & 0xFFFFu)));
    const float dm = __half2float(__ushort_as_half((unsigned short)(hdr.x >> 16)));
    const float rr = ((hdr.x & 0x7FFFu) ? dm / d : dm) * __int_as_float((127 - e) << 23);
    uint32_t sv[4], hv[4], lv[4];
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
        uint32_t sc0, m0, sc1, m1;
        q4k_scale_min(hdr.y, hdr.z, hdr.w, j, sc0, m0);
        q4k_scale_min(hdr.y, hdr.z, hdr.w, j + 1, sc1, m1);
        sv[j >> 1] = h2_bits(__floats2half2_rn((float)sc0 * wmul, (float)sc1 * wmul));
        const float v0 = -rr * (float)m0, v1 = -rr * (float)m1;
        const __half2 hh = __floats2half2_rn(v0, v1);
        const float2 hb = __half22float2(hh);
        hv[j >> 1] = h2_bits(hh);
        lv[j >> 1] = h2_bits(__floats2half2_rn(v0 - hb.x, v1 - hb.y));
    }
    *reinterpret_cast<uint4 *>(srow) = make_uint4(sv[0], sv[1], sv[2], sv[3]);
    const int s32 = (r >> 2) & 1;
    *reinterpret_cast<uint4 *>(mrow + ((0 ^ s32) << 4)) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
    *reinterpret_cast<uint4 *>(mrow + ((1 ^ s32) << 4)) = make_uint4(lv[0], lv[1], lv[2], lv[3]);
    return ((hdr.x & 0x7FFFu) ? d : 1.0f) * __int_as_float((127 + e) << 23);
}

// Converts stage I (nibble bytes 32 I .. 32 I + 31: sub-blocks 2I, low
// nibbles, and 2I + 1, high nibbles) of one weight row to binary16
// sc * q * 2^-e and stores it in the row's TMEM lane at columns col ..
// col + 31 (binary16 pairs in K order: sub-block 2I's 32 weights, then
// 2I + 1's).  s01: the two sub-blocks' scales as binary16 (2I low, 2I + 1
// high).  Low nibble in the mantissa of 1024: s * (1024 + q) - 1024 s; high
// nibble as 1024 + 16 q: (s / 16) * (1024 + 16 q) - 64 s (every step exact).
__device__ __forceinline__ void convert_stage(const uint8_t *raw, int I, uint32_t s01, uint32_t col)
{
    const uint4 n0 = *reinterpret_cast<const uint4 *>(raw + 16 + 32 * I);
    const uint4 n1 = *reinterpret_cast<const uint4 *>(raw + 32 + 32 * I);
    const uint32_t wv[8] = {n0.x, n0.y, n0.z, n0.w, n1.x, n1.y, n1.z, n1.w};
    const __half2 s2 = *reinterpret_cast<const __half2 *>(&s01);
    const __half2 a0 = __low2half2(s2), sh = __high2half2(s2);
    const __half2 b0 = __hmul2(a0, __float2half2_rn(-1024.0f));
    const __half2 a1 = __hmul2(sh, __float2half2_rn(0.0625f)), b1 = __hmul2(sh, __float2half2_rn(-64.0f));
    uint32_t o[32];
#pragma unroll
    for (int c = 0; c < 8; ++c) {   // nibble bytes 4c..4c+3 -> columns 2c, 2c+1 of each sub-block
        const uint32_t p0 = __byte_perm(wv[c], 0, 0x4140), p1 = __byte_perm(wv[c], 0, 0x4342);
        const uint32_t l0 = (p0 & 0x000F000Fu) | 0x64006400u, l1 = (p1 & 0x000F000Fu) | 0x64006400u;
        const uint32_t u0 = (p0 & 0x00F000F0u) | 0x64006400u, u1 = (p1 & 0x00F000F0u) | 0x64006400u;
        o[2 * c] = h2_bits(__hfma2(*reinterpret_cast<const __half2 *>(&l0), a0, b0));
        o[2 * c + 1] = h2_bits(__hfma2(*reinterpret_cast<const __half2 *>(&l1), a0, b0));
        o[16 + 2 * c] = h2_bits(__hfma2(*reinterpret_cast<const __half2 *>(&u0), a1, b1));
        o[16 + 2 * c + 1] = h2_bits(__hfma2(*reinterpret_cast<const __half2 *>(&u1), a1, b1));
    }
    tmem_st32(col, o);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
q4k_gemm_chunk_kernel(const __grid_constant__ CUtensorMap tmap_w, const ChunkParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);

    uint64_t *bm = reinterpret_cast<uint64_t *>(sm + Smem::bars());
    // afull[a]: the weights of super-block l (a = l % 3) are in both CTAs'
    // tensor memory; aempty[a]: its MMAs completed (frees A slot a and min
    // slot a); tok_full[ts] / tok_empty[ts]: the token tiles of a
    // super-block (slot ts) landed in both CTAs / its MMAs completed
    uint64_t *afull = bm, *aempty = afull + kASB;
    uint64_t *raw_full = aempty + kASB, *raw_empty = raw_full + kRawSlots;
    uint64_t *tfull = raw_empty + kRawSlots, *tempty = tfull + kAcc;
    uint64_t *tok_full = tempty + kAcc, *tok_empty = tok_full + kTokSB, *drain = tok_empty + kTokSB;
    // meta_full[m]: the rows' scales, min operand and fold of super-block l
    // (m = l % 6) are in this CTA's shared memory; meta_empty[m]: its
    // epilogue has read the folds (after its MMAs completed), freeing slot m
    uint64_t *meta_full = drain + 1, *meta_empty = meta_full + kMetaSlots;
    // tok_land[ts] (odd CTA): its token copies of slot ts have landed
    uint64_t *tok_land = meta_empty + kMetaSlots;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + Smem::tmem_slot());

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const int pair = blockIdx.x >> 1, P = gridDim.x >> 1;
    const long long g0 = range_start(pair, p.total, P);
    const int L = (int)(range_start(pair + 1, p.total, P) - g0);   // super-blocks of this pair

    if (threadIdx.x == 0) {
        for (int a = 0; a < kASB; ++a) {
            mbar_init(&afull[a], kConvWarps);   // the even CTA's converter warps (+ the odd CTA's st.async bytes)
            mbar_init(&aempty[a], 1);
        }
        for (int ts = 0; ts < kTokSB; ++ts) {
            // the token warp's 32 lanes, each once its copies landed (+ in the
            // even CTA the odd CTA's st.async bytes)
            mbar_init(&tok_full[ts], 32);
            mbar_init(&tok_empty[ts], 1);
            mbar_init(&tok_land[ts], 32);
        }
        for (int i = 0; i < kRawSlots; ++i) {
            mbar_init(&raw_full[i], 1);
            mbar_init(&raw_empty[i], kConvWarps + kMetaWarps);
        }
        for (int m = 0; m < kMetaSlots; ++m) {
            mbar_init(&meta_full[m], kMetaWarps);
            mbar_init(&meta_empty[m], kEpiWarps);
        }
        for (int j = 0; j < kAcc; ++j) {
            mbar_init(&tfull[j], 1);
            mbar_init(&tempty[j], kEpiWarps);
        }
        mbar_init(drain, 1);
        s_abort = 0;
        s_status = p.status;
        fence_mbar_init();
        pdl_launch_dependents();
    }
    if (rank != 0) {
        // the odd CTA's s8 slots are the zero rows (lo columns) of the min MMA's B
        for (int i = threadIdx.x; i < kTokSB * kBMinAtom / 16; i += kThreads)
            reinterpret_cast<uint4 *>(sm + Smem::bmin(0))[i] = make_uint4(0, 0, 0, 0);
        fence_async_smem();
    }
    if (warp == 1) tmem_alloc_pair(tmem_slot, kTmemCols);
    tc_fence_before();
    cluster_sync();   // barriers initialised, zero rows written, tensor memory allocated in both CTAs
    tc_fence_after();
    const PairCtx ctx = pair_ctx(rank);

    if (warp == 0) {
        // -------------------------------------------------- token tiles
        // The whole warp copies each super-block's token tiles (four 16 x 64
        // stages, hi in the even CTA, lo in the odd, 128-byte swizzle; and
        // in the even CTA the s8 tile) into its slot of a ring of kTokSB
        // super-blocks with cp.async.  Each lane's arrival on the slot's
        // barrier follows its copies by hardware, so the warp never waits
        // for a copy, only for a free slot: under full HBM load a copy takes
        // ~3-4 us, and through the TMA unit it would also wait behind the raw
        // tiles.  The odd CTA's slots complete locally (tok_land); its warp 1
        // forwards each to the even CTA's tok_full.
        const __half *src = rank == 0 ? p.hi : p.lo;
        // the tokens may come from the previous kernel on the stream
        // (programmatic launch): wait for it; weights and set-up do not
        pdl_wait();
        bool ok = true;
        for (int l = 0; l < L && ok; ++l) {
            const int ts = l % kTokSB;
            if (l >= kTokSB && !(ok = pair_warp_wait(&tok_empty[ts], ((l / kTokSB) - 1) & 1, ctx))) break;
            // the odd CTA's forwarded signal, counted in bytes
            if (rank == 0 && lane == 0) mbar_expect_tx(&tok_full[ts], kTokSigTx);
            const int b = (int)((g0 + l) % p.nb);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint8_t *dst = sm + Smem::tok(ts, i);
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int c = lane + 32 * m, t = c >> 3, ch = c & 7;   // token row, 16-byte chunk
                    const __half *g = src + (size_t)(t < p.B ? t : 0) * p.K + 256 * b + 64 * i + 8 * ch;
                    cp_async16(dst + 128 * t + ((ch ^ (t & 7)) << 4), g, t < p.B ? 16u : 0u);
                }
            }
            if (rank == 0) {
                // the super-block's s8 tile: 16 rows x 32 bytes, 32-byte swizzle
                const int t = lane >> 1, ch = lane & 1;
                const __half *g = p.s8x + (size_t)(t < p.B ? t : 0) * (p.K / 16) + 16 * b + 8 * ch;
                cp_async16(sm + Smem::bmin(ts) + 32 * t + ((ch ^ ((t >> 2) & 1)) << 4), g, t < p.B ? 16u : 0u);
            }
            cp_async_mbar_arrive(rank == 0 ? &tok_full[ts] : &tok_land[ts]);
        }
        cp_async_wait<0>();   // no copy in flight when the pair tears down
    } else if (warp == 2) {
        // (a warp of its own: a lane of the token producer's warp waiting
        // on the raw ring would hold that warp's token copies back)
        if (lane == 0) {
            // ---------------------------------------------- raw Q4_K tiles
            prefetch_tmap(&tmap_w);
            for (int l = 0; l < L; ++l) {
                const int slot = l % kRawSlots, use = l / kRawSlots;
                if (use > 0 && !pair_wait(&raw_empty[slot], (use - 1) & 1, ctx)) break;
                const long long g = g0 + l;
                const int tile = (int)(g / p.nb), b = (int)(g % p.nb);
                mbar_arrive_expect_tx(&raw_full[slot], (uint32_t)kRawBytes);
                tma_load_2d(sm + Smem::raw(slot), &tmap_w, kQ4KBlockBytes * b, tile * kPairM + kRows * (int)rank,
                            &raw_full[slot]);
            }
        }
    } else if (warp == 1) {
        if (rank != 0) {
            // ------------------------- odd CTA: forward landed token slots
            const uint32_t sig = cluster_addr(smem_u32(sm + Smem::sig()) + 4u * (kConvWarps + kEpiWarps), 0);
            static_assert(4 * (kConvWarps + kEpiWarps + 2) <= 128, "st.async words of the odd CTA's warps");
            const uint32_t tfull_cl0 = cluster_addr(smem_u32(&tok_full[0]), 0);
            for (int l = 0; l < L; ++l) {
                const int ts = l % kTokSB;
                if (!pair_warp_wait(&tok_land[ts], (uint32_t)(l / kTokSB) & 1u, ctx)) break;
                fence_async_smem();   // the MMA reads the copies through the async proxy
                if (lane == 0) st_async_signal(sig, tfull_cl0 + 8u * (uint32_t)ts);
            }
        }
        // ---------------------------------------------------- MMA issuer
        // (the whole warp runs the loop and waits; one elected lane issues)
        if (rank == 0) {
            const uint32_t tmem = *tmem_slot;
            const uint32_t base = smem_u32(sm);
            const uint64_t bt0 = smem_desc(base + (uint32_t)Smem::tok(0, 0), 16, 1024, kLayoutSw128);
            const uint64_t bmn = smem_desc(base + (uint32_t)Smem::bmin(0), 16, 256, kLayoutSw32);
            const uint64_t amn = smem_desc(base + (uint32_t)Smem::amin(0), 16, 256, kLayoutSw32);
            constexpr uint64_t kT16 = kTokAtom >> 4, kBM16 = kBMinAtom >> 4, kAM16 = kAMinAtom >> 4;
            constexpr uint32_t idesc = idesc_f16_f32(kPairM, kN);
            bool ok = true;
            for (int l = 0; l < L && ok; ++l) {
                const int j = l % kAcc, ts = l % kTokSB, a = l % kASB, m = l % kMetaSlots;
                // the epilogues have read accumulator j (super-block l - 4)
                if (l >= kAcc && !(ok = __all_sync(0xffffffffu, pair_wait(&tempty[j], ((l / kAcc) - 1) & 1, ctx))))
                    break;
                // the super-block's token tiles and converted weights are in both CTAs
                if (!(ok = __all_sync(0xffffffffu, pair_wait(&tok_full[ts], (l / kTokSB) & 1, ctx)))) break;
                if (!(ok = __all_sync(0xffffffffu, pair_wait(&afull[a], (l / kASB) & 1, ctx)))) break;
                fence_async_smem();   // this CTA's token copies landed (cp.async): order them before the MMAs
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(kN * j);
                const uint32_t a_tmem = tmem + kACol0 + kACols * a;
                const uint64_t bt = bt0 + (uint64_t)(4 * ts) * kT16;
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < 16; ++kk)   // K = 16 steps of the super-block
                        mma_f16_pair_ta(d, a_tmem + 8 * kk, bt + (uint64_t)(kk >> 2) * kT16 + 2 * (kk & 3), idesc,
                                        kk != 0 ? 1u : 0u);
                    mma_f16_pair(d, amn + (uint64_t)m * kAM16, bmn + (uint64_t)ts * kBM16, idesc, 1u);
                    mma_commit_pair_mc(&tfull[j], 3);
                    mma_commit_pair_mc(&tok_empty[ts], 3);
                    mma_commit_pair_mc(&aempty[a], 3);
                }
                __syncwarp();
            }
            // every MMA issued has completed before the pair tears down
            if (elect_one()) mma_commit_pair_local(drain);
            __syncwarp();
            drain_wait(drain, 0);
        }
    } else if (warp >= kConvWarp0 && warp < kConvWarp0 + kConvWarps) {
        // ---------------------------------------------------- converters
        const uint32_t tmem = *tmem_slot;
        const int quarter = warp & 3, st = (warp - kConvWarp0) >> 2;   // lane quarter, K = 64 stage
        const int r = 32 * quarter + lane;   // weight row = TMEM lane
        const uint32_t lane_base = tmem + ((uint32_t)(32 * quarter) << 16) + kACol0 + 32u * (uint32_t)st;
        const uint32_t sig = cluster_addr(smem_u32(sm + Smem::sig()) + 4u * (warp - kConvWarp0), 0);
        const uint32_t afull_cl0 = cluster_addr(smem_u32(&afull[0]), 0);   // barriers 8 bytes apart
        bool ok = true;
        // ring positions kept as counters: raw and metadata slot rs (phase
        // rph; both rings have kRawSlots slots), A slot a (phase aph)
        int rs = 0, a = 0;
        uint32_t rph = 0, aph = 0;
        static_assert(kMetaSlots == kRawSlots, "one counter for both rings");
        for (int l = 0; l < L && ok; ++l) {
            if (!(ok = pair_warp_wait(&raw_full[rs], rph, ctx))) break;
            if (!(ok = pair_warp_wait(&meta_full[rs], rph, ctx))) break;   // the rows' scales
            if (l >= kASB && !(ok = pair_warp_wait(&aempty[a], aph ^ 1u, ctx))) break;
            tc_fence_after();
            const uint32_t s01 =
                *reinterpret_cast<const uint32_t *>(sm + Smem::scales(rs) + (size_t)r * kScaleRow + 4 * st);
            convert_stage(sm + Smem::raw(rs) + (size_t)r * kQ4KBlockBytes, st, s01, lane_base + kACols * a);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                signal_leader(&afull[a], rank, quarter == 0 && st == 0, kConvSigTx, sig, afull_cl0 + 8u * (uint32_t)a);
                mbar_arrive(&raw_empty[rs]);
            }
            if (++rs == kRawSlots) { rs = 0; rph ^= 1u; }
            if (++a == kASB) { a = 0; aph ^= 1u; }
        }
    } else if (warp >= kMetaWarp0 && warp < kMetaWarp0 + kMetaWarps) {
        // ----------------------------------------------------- row metadata
        // Super-block l's row metadata (scales, min operand, fold), decoded
        // once its raw tile has landed and the epilogue of l - 6 has
        // released metadata slot l % 6.
        const int r = 32 * (warp & 3) + lane;
        bool ok = true;
        int rs = 0;   // raw and metadata slot (phase rph)
        uint32_t rph = 0;
        for (int l = 0; l < L && ok; ++l) {
            if (!(ok = pair_warp_wait(&raw_full[rs], rph, ctx))) break;
            if (l >= kMetaSlots && !(ok = pair_warp_wait(&meta_empty[rs], rph ^ 1u, ctx))) break;
            const float f = decode_row(sm + Smem::raw(rs) + (size_t)r * kQ4KBlockBytes,
                                       sm + Smem::scales(rs) + (size_t)r * kScaleRow,
                                       sm + Smem::amin(rs) + (size_t)r * 32, r);
            reinterpret_cast<float *>(sm + Smem::fold(rs))[r] = f;
            fence_async_smem();   // the min MMA reads the min operand through the async proxy
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&meta_full[rs]);
                mbar_arrive(&raw_empty[rs]);
            }
            if (++rs == kRawSlots) { rs = 0; rph ^= 1u; }
        }
    } else if (warp >= kEpiWarp0) {
        // ---------------------------------------------------------- epilogue
        pdl_wait();   // y, the partial sums and the token scales
        const uint32_t tmem = *tmem_slot;
        const int quarter = warp & 3;
        const int r = 32 * quarter + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(32 * quarter) << 16);
        const uint32_t sig = cluster_addr(smem_u32(sm + Smem::sig()) + 4u * kConvWarps + 4u * quarter, 0);
        const uint32_t tempty_cl0 = cluster_addr(smem_u32(&tempty[0]), 0);
        float acc[kTok];
#pragma unroll
        for (int t = 0; t < kTok; ++t) acc[t] = 0.0f;
        bool ok = true;
        int ms = 0;   // metadata slot of super-block l
        int etile = (int)(g0 / p.nb), eb = (int)(g0 % p.nb);   // tile and super-block of l
        for (int l = 0; l < L && ok; ++l) {
            const int n = etile * kPairM + kRows * (int)rank + r;
            const bool nvalid = n < p.N;
            const int j = l % kAcc;
            if (!(ok = pair_warp_wait(&tfull[j], (uint32_t)(l / kAcc) & 1, ctx))) break;
            // (the fold was written before the converters, hence the MMAs, of l could start)
            const float fold = nvalid ? reinterpret_cast<const float *>(sm + Smem::fold(ms))[r] : 0.0f;
            tc_fence_after();
            uint32_t v[32];
            tmem_ld32(lane_base + (uint32_t)(kN * j), v);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                signal_leader(&tempty[j], rank, quarter == 0, kEpiSigTx, sig, tempty_cl0 + 8u * (uint32_t)j);
                mbar_arrive(&meta_empty[ms]);
            }
#pragma unroll
            for (int t = 0; t < kTok; ++t)
                acc[t] = fmaf(fold, __uint_as_float(v[t]) + __uint_as_float(v[kTok + t]), acc[t]);
            // the tile's last super-block in this range: write its rows
            if (l == L - 1 || eb + 1 == p.nb) {
                if (nvalid) {
                    const long long t0g = (long long)etile * p.nb;
                    const int pf = pair_of(t0g, p.total, P);
                    const int pl = pair_of(t0g + p.nb - 1, p.total, P);
                    float *out = (pf == pl) ? p.y + n : p.part + ((size_t)(pair - pf) * p.B) * p.N + n;
#pragma unroll
                    for (int t = 0; t < kTok; ++t)
                        if (t < p.B) out[(size_t)t * p.N] = acc[t] * __ldg(p.tscale + t);
                }
#pragma unroll
                for (int t = 0; t < kTok; ++t) acc[t] = 0.0f;
            }
            if (++eb == p.nb) {
                eb = 0;
                ++etile;
            }
            if (++ms == kMetaSlots) ms = 0;
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
    tc_fence_before();
    cluster_sync();   // the peer's MMAs, copies and signals are finished
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(*tmem_slot, kTmemCols);
    }
}

// y[t][n] of the tiles that straddle ranges: the sum of their pieces in
// range order.  Block (tile, t): the tile's 256 rows of token t; the
// tile's first and last pair are found once per block.
__global__ void __launch_bounds__(kPairM) chunk_fixup_kernel(const float *__restrict__ part, int B, int N, int nb,
                                                             long long total, int P, float *__restrict__ y)
{
    __shared__ int s_pf, s_np;
    const int tile = blockIdx.x, t = blockIdx.y;
    if (threadIdx.x == 0) {
        const long long t0g = (long long)tile * nb;
        s_pf = pair_of(t0g, total, P);
        s_np = pair_of(t0g + nb - 1, total, P) - s_pf + 1;
    }
    __syncthreads();
    const int n = tile * kPairM + threadIdx.x;
    if (s_np == 1 || n >= N) return;
    float a = part[(size_t)t * N + n];
    for (int s = 1; s < s_np; ++s) a += part[((size_t)s * B + t) * N + n];
    y[(size_t)t * N + n] = a;
}

size_t g_attr_bytes[64];
int g_max_pairs[64];

// CTA pairs that can be resident at once (a pair needs two SMs of one GPC)
int chunk_pairs(int sms)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return sms / 2;
    }
    if (g_max_pairs[dev] == 0) {
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(2 * (sms / 2));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = Smem::total();
        int n = 0;
        if (cudaFuncSetAttribute(q4k_gemm_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)Smem::total()) != cudaSuccess ||
            cudaOccupancyMaxActiveClusters(&n, q4k_gemm_chunk_kernel, &cfg) != cudaSuccess || n < 1) {
            cudaGetLastError();
            n = sms / 2;
        }
        g_max_pairs[dev] = n < sms / 2 ? n : sms / 2;
    }
    return g_max_pairs[dev];
}

}  // namespace

// Pieces of the largest straddling tile for P pairs (the partial-sum slots
// the workspace needs); 0 when no tile straddles.
static int chunk_pieces(int N, int K, int P)
{
    const int nb = K / 256, tiles = (N + kPairM - 1) / kPairM;
    const long long total = (long long)tiles * nb;
    if (P > total) P = (int)total;
    int most = 0;
    for (int t = 0; t < tiles; ++t) {
        const int pf = pair_of((long long)t * nb, total, P), pl = pair_of((long long)t * nb + nb - 1, total, P);
        if (pl > pf && pl - pf + 1 > most) most = pl - pf + 1;
    }
    return most;
}

// CTA pairs of a launch.  One pair per tile (its whole K range, no partial
// sums) when splitting is not allowed or the tiles already fill the
// resident pairs about as well as balanced ranges would (the fixup launch
// costs about three super-blocks); else as many pairs as can be resident,
// over balanced ranges.
static int chunk_plan(int N, int K, bool allow_split)
{
    const int nb = K / 256, tiles = (N + kPairM - 1) / kPairM;
    const long long total = (long long)tiles * nb;
    const int pmax = chunk_pairs(num_sms());
    const long long waves = (tiles + pmax - 1) / pmax;
    const long long split_cost = (total + pmax - 1) / pmax + 3;
    if (!allow_split || waves * nb <= split_cost) return tiles;
    return pmax < total ? pmax : (int)total;
}

size_t chunk_part_bytes(int N, int K, int B)
{
    const int P = chunk_plan(N, K, true);
    const int tiles = (N + kPairM - 1) / kPairM;
    return P == tiles ? 0 : (size_t)chunk_pieces(N, K, P) * B * N * sizeof(float);
}

cudaError_t launch_gemm_chunk(const void *W, int N, int K, int B, const __half *hi, const __half *lo,
                              const __half *s8x, const float *tscale, float *y, float *part, bool allow_split,
                              cudaStream_t st)
{
    CUtensorMap tw;
    const CUtensorMapDataType u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
    cudaError_t e;
    if ((e = make_tmap_2d(&tw, u8, 1, W, (uint64_t)(K / 256) * kQ4KBlockBytes, (uint64_t)N, kQ4KBlockBytes, kRows,
                          CU_TENSOR_MAP_SWIZZLE_NONE)) != cudaSuccess)
        return e;
    ChunkParams p{};
    p.N = N;
    p.K = K;
    p.B = B;
    p.nb = K / 256;
    p.tiles = (N + kPairM - 1) / kPairM;
    p.total = (long long)p.tiles * p.nb;
    p.row_bytes = (size_t)p.nb * kQ4KBlockBytes;
    p.W = static_cast<const uint8_t *>(W);
    p.tscale = tscale;
    p.hi = hi;
    p.lo = lo;
    p.s8x = s8x;
    p.y = y;
    p.part = part;
    p.status = device_status_word();
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    const size_t smem = Smem::total();
    if (g_attr_bytes[dev] < smem) {
        e = cudaFuncSetAttribute(q4k_gemm_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        g_attr_bytes[dev] = smem;
    }
    const int P = chunk_plan(N, K, allow_split);
    if ((e = launch_pdl(q4k_gemm_chunk_kernel, dim3((unsigned)(2 * P)), dim3(kThreads), smem, st, tw, p)) !=
        cudaSuccess)
        return e;
    if (P == p.tiles || chunk_pieces(N, K, P) == 0) return cudaSuccess;
    chunk_fixup_kernel<<<dim3(p.tiles, B), kPairM, 0, st>>>(part, B, N, p.nb, p.total, P, y);
    return cudaGetLastError();
}

}  // namespace zq
