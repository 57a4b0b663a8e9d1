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
// weight rows, K = 32 as two K = 16 steps) writes one of four TMEM buffers
// (all 512 columns); epilogue warps read it back and fold it into an fp32
// accumulator held in registers, acc += d_b * (d8 * D) (d8 is a per-lane
// scalar: TMEM lanes are tokens; d_b a per-column one).  Once per super-block
// a second MMA forms sum_j s8[t][bj] * m_j[n] (K = 16: eight mins and eight
// zeros) in a buffer of the same ring, and the epilogue subtracts
// dmin_b * minsum.
//
// Warp roles (20 warps): 0 TMA producer (fp16 activation tiles in a
// six-stage ring, s8 tiles, raw Q4_K tiles two super-blocks ahead), 1 MMA
// issuer + TMEM owner, 2-3 weight converters (Q4_K bytes -> sc*q fp16 in the
// 128-byte-swizzled K-major layout, two rows per thread, three-stage ring;
// mins; d/dmin), 4-19 epilogue (4 column groups of 32 x 4 lane quarters),
// which hand each TMEM buffer back right after reading it.  The issuer keeps
// its loop to descriptor additions and counter updates: one thread feeds the
// tensor pipe, so its instruction count per MMA bounds the kernel.  Every
// wait is bounded.
#include <cuda.h>

#include "zq_internal.cuh"
#include "zq_tc.cuh"

namespace zq {
namespace {

constexpr int BM = 128;               // tokens per tile (TMEM lanes)
constexpr int BN = 128;               // weight rows per tile (TMEM columns)
constexpr int kAStages = 6;           // activation operand stages of K = 64 (two sub-blocks)
constexpr int kBStages = 3;           // converted weight operand stages of K = 64
constexpr int kAtomBytes = 128 * 128; // 128 rows x 64 fp16 (128 B), 128-byte swizzle
constexpr int kRawSlots = 3;          // raw Q4_K tiles in flight (super-blocks)
constexpr int kRawBytes = BN * kQ4KBlockBytes;  // 128 rows x 144 B
constexpr int kMinBytes = 128 * 32;   // 128 rows x 16 fp16, 32-byte swizzle
constexpr int kRing = 4;              // TMEM result buffers (sub-block or min products)
constexpr int kWarps = 20;
constexpr int kThreads = kWarps * 32;
constexpr int kConvWarp0 = 2, kConvWarps = 2;   // each converter thread owns two weight rows
constexpr int kEpiWarp0 = 4, kEpiWarps = 16;
constexpr int kEpiCols = BN / (kEpiWarps / 4);   // 32 columns per epilogue thread
constexpr uint32_t kIdesc = idesc_f16_f32(BM, BN);
constexpr uint32_t kTmemCols = 512;
static_assert(kRing * BN == (int)kTmemCols, "the result ring fills tensor memory");
static_assert((kRing & (kRing - 1)) == 0, "ring index by mask");

struct Smem {
    // offsets from the 1024-aligned base
    static constexpr size_t a_atom(int s) { return (size_t)s * kAtomBytes; }
    static constexpr size_t b_atom(int s) { return a_atom(kAStages) + (size_t)s * kAtomBytes; }
    static constexpr size_t raw(int i) { return b_atom(kBStages) + (size_t)i * kRawBytes; }
    static constexpr size_t amin(int i) { return raw(kRawSlots) + (size_t)i * 2 * kMinBytes; }
    static constexpr size_t bmin(int i) { return amin(i) + kMinBytes; }
    static constexpr size_t dd(int i) { return amin(2) + (size_t)i * BN * 8; }  // d[BN] then dmin[BN]
    static constexpr size_t bars() { return dd(2); }
    static constexpr int kNumBars = 2 * kAStages + 2 * kBStages + 2 * kRawSlots + 3 * 2 + 2 * kRing + 2 * 2;
    static constexpr size_t tmem_slot() { return bars() + kNumBars * 8; }
    static constexpr size_t total() { return tmem_slot() + 16 + 1024; }  // + alignment slack
};
static_assert(Smem::total() <= 227 * 1024, "shared memory budget");
static_assert(kRawBytes % 1024 == 0, "raw slots keep the operand atoms 1024-byte aligned");
static_assert(Smem::total() < (1u << 18), "descriptor start addresses stay inside their 14-bit field");

struct Bars {
    uint64_t *a_full, *a_empty;                   // [kAStages]
    uint64_t *b_full, *b_empty;                   // [kBStages]
    uint64_t *raw_full, *raw_empty;               // [kRawSlots]
    uint64_t *amin_full, *bmin_full, *min_empty;  // [2]
    uint64_t *ring_full, *ring_empty;             // [kRing]
    uint64_t *dd_full, *dd_free;                  // [2]
};

struct GemmParams {
    int N, K, B, nb;
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

// (c0, c1) += (d0, d1) * ((a0, a1) * (s, s)): two packed fp32x2 operations
__device__ __forceinline__ void scale_acc2(float &c0, float &c1, float a0, float a1, float s, float d0, float d1)
{
    asm("{\n\t.reg .b64 ra, rs, rd, rc;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rs, {%4, %4};\n\tmov.b64 rd, {%5, %6};\n\tmov.b64 rc, {%0, %1};\n\t"
        "mul.rn.f32x2 ra, ra, rs;\n\tfma.rn.f32x2 rc, rd, ra, rc;\n\tmov.b64 {%0, %1}, rc;\n\t}"
        : "+f"(c0), "+f"(c1)
        : "f"(a0), "f"(a1), "f"(s), "f"(d0), "f"(d1));
}

// bounded wait that also gives up at once when another role already failed
__device__ __noinline__ bool wait_ok(uint64_t *bar, uint32_t parity, volatile int *abort_flag, unsigned int *status)
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

// one probe inline, the bounded loop only when the phase is not complete yet
__device__ __forceinline__ bool wait_fast(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                          unsigned int *status)
{
    return mbar_try_wait(bar, parity) || wait_ok(bar, parity, abort_flag, status);
}

// one lane polls, then every lane acquires the completed phase itself
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                         unsigned int *status)
{
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = wait_fast(bar, parity, abort_flag, status);
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    if (ok) ok = wait_fast(bar, parity, abort_flag, status);
    return __all_sync(0xffffffffu, ok);
}

template <bool DEBUG>
__global__ void __maxnreg__(96)
q4k_gemm_wide_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_s,
                     const __grid_constant__ CUtensorMap tmap_w, const GemmParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    __shared__ volatile int abort_s;

    uint64_t *bm = reinterpret_cast<uint64_t *>(sm + Smem::bars());
    Bars bar;
    bar.a_full = bm;
    bar.a_empty = bar.a_full + kAStages;
    bar.b_full = bar.a_empty + kAStages;
    bar.b_empty = bar.b_full + kBStages;
    bar.raw_full = bar.b_empty + kBStages;
    bar.raw_empty = bar.raw_full + kRawSlots;
    bar.amin_full = bar.raw_empty + kRawSlots;
    bar.bmin_full = bar.amin_full + 2;
    bar.min_empty = bar.bmin_full + 2;
    bar.ring_full = bar.min_empty + 2;
    bar.ring_empty = bar.ring_full + kRing;
    bar.dd_full = bar.ring_empty + kRing;
    bar.dd_free = bar.dd_full + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + Smem::tmem_slot());

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int t_tile = blockIdx.x % p.t_tiles;
    const int n_tile = blockIdx.x / p.t_tiles;
    const int t0 = t_tile * BM;
    const int n0 = n_tile * BN;
    const int nb = p.nb;
    const int nq = 4 * nb;   // operand stages (K = 64 each)
    // Each CTA walks the super-blocks in its own rotated order, so the CTAs
    // that share an activation tile (and those that share a weight tile) do not
    // all request the same L2 lines at the same time.  The fp32 sums are
    // order-free; the integer sub-block sums are unaffected.
    const int rot = (n_tile + 5 * t_tile) % nb;
    auto sb = [&](int b) { return b + rot < nb ? b + rot : b + rot - nb; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kAStages; ++s) {
            mbar_init(&bar.a_full[s], 1);
            mbar_init(&bar.a_empty[s], 1);
        }
        for (int s = 0; s < kBStages; ++s) {
            mbar_init(&bar.b_full[s], kConvWarps);
            mbar_init(&bar.b_empty[s], 1);
        }
        for (int s = 0; s < kRawSlots; ++s) {
            mbar_init(&bar.raw_full[s], 1);
            mbar_init(&bar.raw_empty[s], kConvWarps);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar.amin_full[i], 1);
            mbar_init(&bar.bmin_full[i], kConvWarps);
            mbar_init(&bar.min_empty[i], 1);
            mbar_init(&bar.dd_full[i], kConvWarps);
            mbar_init(&bar.dd_free[i], kEpiWarps);
        }
        for (int i = 0; i < kRing; ++i) {
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
            prefetch_tmap(&tmap_a);
            prefetch_tmap(&tmap_s);
            prefetch_tmap(&tmap_w);
            bool ok = true;
            // raw weight tiles run kRawSlots - 1 super-blocks ahead of the
            // activation tiles; activation stage q = 4b + i
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
                const int slot = q % kAStages, round = q / kAStages;
                if (round > 0 && !(ok = wait_fast(&bar.a_empty[slot], (round - 1) & 1, &abort_s, p.status))) break;
                mbar_arrive_expect_tx(&bar.a_full[slot], kAtomBytes);
                tma_load_2d(sm + Smem::a_atom(slot), &tmap_a, 256 * sb(b) + 64 * i, t0, &bar.a_full[slot]);
                if (i == 0) {
                    const int mi = b & 1, use = b >> 1;
                    if (use > 0 && !(ok = wait_fast(&bar.min_empty[mi], (use - 1) & 1, &abort_s, p.status))) break;
                    mbar_arrive_expect_tx(&bar.amin_full[mi], kMinBytes);
                    tma_load_2d(sm + Smem::amin(mi), &tmap_s, 8 * sb(b), t0, &bar.amin_full[mi]);
                }
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t base = smem_u32(sm);
            // descriptors of stage 0 / min slot 0; every other operand tile is
            // reached by adding its byte offset / 16 to the start-address field
            const uint64_t a_desc0 = smem_desc(base + (uint32_t)Smem::a_atom(0), 16, 1024, kLayoutSw128);
            const uint64_t b_desc0 = smem_desc(base + (uint32_t)Smem::b_atom(0), 16, 1024, kLayoutSw128);
            const uint64_t amin_desc0 = smem_desc(base + (uint32_t)Smem::amin(0), 16, 256, kLayoutSw32);
            const uint64_t bmin_desc0 = smem_desc(base + (uint32_t)Smem::bmin(0), 16, 256, kLayoutSw32);
            constexpr uint32_t kAtom16 = kAtomBytes >> 4, kMinSlot16 = (2 * kMinBytes) >> 4;
            int as = 0, bs = 0;
            uint32_t aph = 0, bph = 0, e = 0;   // e: ring entries issued so far
            bool ok = true;
            for (int b = 0; b < nb && ok; ++b) {
                for (int i = 0; i < 4; ++i) {
                    if (!(ok = wait_fast(&bar.a_full[as], aph, &abort_s, p.status) &&
                               wait_fast(&bar.b_full[bs], bph, &abort_s, p.status)))
                        break;
                    const uint64_t ad = a_desc0 + (uint64_t)(as * kAtom16);
                    const uint64_t bd = b_desc0 + (uint64_t)(bs * kAtom16);
#pragma unroll
                    for (int jj = 0; jj < 2; ++jj, ++e) {
                        const uint32_t buf = e & (kRing - 1);
                        if (e >= (uint32_t)kRing &&
                            !(ok = wait_fast(&bar.ring_empty[buf], ((e / kRing) - 1) & 1, &abort_s, p.status)))
                            break;
                        tc_fence_after();
                        const uint32_t d_tmem = tmem + (uint32_t)BN * buf;
                        mma_f16(d_tmem, ad + (uint64_t)(jj * 4), bd + (uint64_t)(jj * 4), kIdesc, 0u);
                        mma_f16(d_tmem, ad + (uint64_t)(jj * 4 + 2), bd + (uint64_t)(jj * 4 + 2), kIdesc, 1u);
                        mma_commit(&bar.ring_full[buf]);
                    }
                    if (!ok) break;
                    mma_commit(&bar.a_empty[as]);
                    mma_commit(&bar.b_empty[bs]);
                    if (++as == kAStages) { as = 0; aph ^= 1u; }
                    if (++bs == kBStages) { bs = 0; bph ^= 1u; }
                }
                if (!ok) break;
                // the super-block's min product: sum_j s8[t][bj] * m_j[n]
                const int mi = b & 1;
                const uint32_t mpar = (uint32_t)(b >> 1) & 1u, buf = e & (kRing - 1);
                if (!(ok = wait_fast(&bar.amin_full[mi], mpar, &abort_s, p.status) &&
                           wait_fast(&bar.bmin_full[mi], mpar, &abort_s, p.status) &&
                           (e < (uint32_t)kRing ||
                            wait_fast(&bar.ring_empty[buf], ((e / kRing) - 1) & 1, &abort_s, p.status))))
                    break;
                tc_fence_after();
                mma_f16(tmem + (uint32_t)BN * buf, amin_desc0 + (uint64_t)(mi * kMinSlot16),
                        bmin_desc0 + (uint64_t)(mi * kMinSlot16), kIdesc, 0u);
                mma_commit(&bar.ring_full[buf]);
                mma_commit(&bar.min_empty[mi]);
                ++e;
            }
        }
    } else if (warp < kEpiWarp0) {
        // ---------------------------------------------------- converters
        // thread r converts weight rows r and r + 64 of the tile
        const int r0 = (warp - kConvWarp0) * 32 + lane;
        for (int b = 0; b < nb; ++b) {
            const int rs = b % kRawSlots, ruse = b / kRawSlots;
            if (!warp_wait(&bar.raw_full[rs], ruse & 1, &abort_s, p.status)) break;
            const uint8_t *rawbase = sm + Smem::raw(rs);
            const uint4 hdr0 = *reinterpret_cast<const uint4 *>(rawbase + (size_t)r0 * kQ4KBlockBytes);
            const uint4 hdr1 = *reinterpret_cast<const uint4 *>(rawbase + (size_t)(r0 + 64) * kQ4KBlockBytes);
            bool ok = true;
            for (int i = 0; i < 4 && ok; ++i) {
                const int q = 4 * b + i;
                const int bs = q % kBStages, round = q / kBStages;
                if (round > 0 && !(ok = warp_wait(&bar.b_empty[bs], (round - 1) & 1, &abort_s, p.status))) break;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int r = r0 + 64 * h;
                    const uint4 &hdr = h ? hdr1 : hdr0;
                    const uint8_t *raw = rawbase + (size_t)r * kQ4KBlockBytes;
                    const uint4 n0v = *reinterpret_cast<const uint4 *>(raw + 16 + 32 * i);
                    const uint4 n1v = *reinterpret_cast<const uint4 *>(raw + 32 + 32 * i);
                    uint32_t sc0, sc1, md;
                    q4k_scale_min(hdr.y, hdr.z, hdr.w, 2 * i, sc0, md);
                    q4k_scale_min(hdr.y, hdr.z, hdr.w, 2 * i + 1, sc1, md);
                    const float scl = DEBUG ? 1.0f : (float)sc0;
                    const float sch = DEBUG ? 1.0f : (float)sc1;
                    const __half2 s_lo = __float2half2_rn(scl), o_lo = __float2half2_rn(-1024.0f * scl);
                    const __half2 s_hi = __float2half2_rn(sch * 0.0625f), o_hi = __float2half2_rn(-64.0f * sch);
                    const uint32_t wv[8] = {n0v.x, n0v.y, n0v.z, n0v.w, n1v.x, n1v.y, n1v.z, n1v.w};
                    uint8_t *atom = sm + Smem::b_atom(bs) + (size_t)r * 128;
                    const int sw = r & 7;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint4 lo, hi;
                        nib4_to_h2<false>(wv[2 * c], s_lo, o_lo, lo.x, lo.y);
                        nib4_to_h2<false>(wv[2 * c + 1], s_lo, o_lo, lo.z, lo.w);
                        nib4_to_h2<true>(wv[2 * c], s_hi, o_hi, hi.x, hi.y);
                        nib4_to_h2<true>(wv[2 * c + 1], s_hi, o_hi, hi.z, hi.w);
                        *reinterpret_cast<uint4 *>(atom + ((c ^ sw) << 4)) = lo;
                        *reinterpret_cast<uint4 *>(atom + (((c + 4) ^ sw) << 4)) = hi;
                    }
                }
                if (i == 0) {
                    const int mi = b & 1, use = b >> 1;
                    // mins as the B operand of the min MMA; d, dmin for the epilogue
                    if (use > 0 && !(ok = warp_wait(&bar.min_empty[mi], (use - 1) & 1, &abort_s, p.status))) break;
                    if (use > 0 && !(ok = warp_wait(&bar.dd_free[mi], (use - 1) & 1, &abort_s, p.status))) break;
                    float *ddp = reinterpret_cast<float *>(sm + Smem::dd(mi));
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int r = r0 + 64 * h;
                        const uint4 &hdr = h ? hdr1 : hdr0;
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
                        ddp[r] = dm.x;
                        ddp[BN + r] = dm.y;
                    }
                    fence_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&bar.bmin_full[mi]);
                        mbar_arrive(&bar.dd_full[mi]);
                    }
                }
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar.b_full[bs]);
            }
            if (!ok) break;
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar.raw_empty[rs]);
        }
    } else {
        // ---------------------------------------------------- epilogue
        const int e_w = warp - kEpiWarp0;
        const int cg = e_w >> 2;                  // column group: columns 32cg .. 32cg+31
        const int quarter = warp & 3;             // TMEM lanes 32*quarter .. +31
        const int tl = 32 * quarter + lane;       // token within the tile
        const int tok = t0 + tl;
        const bool tvalid = tok < p.B;
        const uint32_t lane_base = tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(kEpiCols * cg);
        const int nsub = nb * 8;
        float acc[kEpiCols];
#pragma unroll
        for (int c = 0; c < kEpiCols; ++c) acc[c] = 0.0f;
        uint4 d8raw = make_uint4(0, 0, 0, 0);
        if (tvalid && !DEBUG) d8raw = __ldg(reinterpret_cast<const uint4 *>(p.d8 + (size_t)tok * nsub + 8 * sb(0)));
        bool ok = true;
        uint32_t e = 0;   // ring entries consumed so far
        for (int b = 0; b < nb && ok; ++b) {
            const int mi = b & 1, muse = b >> 1;
            uint4 d8next = make_uint4(0, 0, 0, 0);
            if (tvalid && !DEBUG && b + 1 < nb)
                d8next = __ldg(reinterpret_cast<const uint4 *>(p.d8 + (size_t)tok * nsub + 8 * sb(b + 1)));
            if (!(ok = warp_wait(&bar.dd_full[mi], muse & 1, &abort_s, p.status))) break;
            const float *dcol = reinterpret_cast<const float *>(sm + Smem::dd(mi)) + kEpiCols * cg;
            for (int j = 0; j < 9; ++j, ++e) {   // j = 8: the min product
                const uint32_t buf = e & (kRing - 1);
                if (!(ok = warp_wait(&bar.ring_full[buf], (e / kRing) & 1, &abort_s, p.status))) break;
                tc_fence_after();
                uint32_t r[32];
                tmem_ld32(lane_base + (uint32_t)BN * buf, r);
                tmem_wait_ld();
                // hand the buffer back before the arithmetic
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar.ring_empty[buf]);
                if (DEBUG) {
                    if (tvalid && j < 8) {
#pragma unroll
                        for (int c = 0; c < 32; ++c) {
                            const int n = n0 + kEpiCols * cg + c;
                            if (n < p.N)
                                p.isums[((size_t)tok * p.N + n) * nsub + 8 * sb(b) + j] = (int32_t)__uint_as_float(r[c]);
                        }
                    }
                } else if (j < 8) {
                    const uint32_t w2 = (j < 4) ? ((j < 2) ? d8raw.x : d8raw.y) : ((j < 6) ? d8raw.z : d8raw.w);
                    const uint16_t hb = (j & 1) ? (uint16_t)(w2 >> 16) : (uint16_t)(w2 & 0xFFFFu);
                    const float d8 = __half2float(__ushort_as_half(hb));
#pragma unroll
                    for (int c = 0; c < 32; c += 4) {
                        const float4 dv = *reinterpret_cast<const float4 *>(dcol + c);
                        scale_acc2(acc[c], acc[c + 1], __uint_as_float(r[c]), __uint_as_float(r[c + 1]), d8, dv.x, dv.y);
                        scale_acc2(acc[c + 2], acc[c + 3], __uint_as_float(r[c + 2]), __uint_as_float(r[c + 3]), d8,
                                   dv.z, dv.w);
                    }
                } else {
                    // super-block end: acc -= dmin_b * minsum
#pragma unroll
                    for (int c = 0; c < 32; c += 4) {
                        const float4 mv = *reinterpret_cast<const float4 *>(dcol + BN + c);
                        acc[c] = fmaf(-mv.x, __uint_as_float(r[c]), acc[c]);
                        acc[c + 1] = fmaf(-mv.y, __uint_as_float(r[c + 1]), acc[c + 1]);
                        acc[c + 2] = fmaf(-mv.z, __uint_as_float(r[c + 2]), acc[c + 2]);
                        acc[c + 3] = fmaf(-mv.w, __uint_as_float(r[c + 3]), acc[c + 3]);
                    }
                }
            }
            if (!ok) break;
            d8raw = d8next;
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar.dd_free[mi]);
        }
        if (ok && !abort_s && !DEBUG && tvalid) {
            float *yrow = p.y + (size_t)tok * p.N + n0 + kEpiCols * cg;
            const int ncols = min(kEpiCols, p.N - (n0 + kEpiCols * cg));
            if (ncols == kEpiCols && (p.N & 3) == 0) {
#pragma unroll
                for (int c = 0; c < kEpiCols; c += 4)
                    *reinterpret_cast<float4 *>(yrow + c) = make_float4(acc[c], acc[c + 1], acc[c + 2], acc[c + 3]);
            } else {
#pragma unroll
                for (int c = 0; c < kEpiCols; ++c)
                    if (c < ncols) yrow[c] = acc[c];
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

// 2-D tensor [rows][cols] of `esize`-byte elements, row stride = cols*esize
// bytes, box box_cols x box_rows; out-of-range elements read as zero
cudaError_t make_tmap(CUtensorMap *m, CUtensorMapDataType dt, uint32_t esize, const void *base, uint64_t cols,
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
    CUtensorMap ta, ts, tw;
    const CUtensorMapDataType f16 = CU_TENSOR_MAP_DATA_TYPE_FLOAT16, u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
    if ((e = make_tmap(&ta, f16, 2, a16, (uint64_t)K, (uint64_t)B, 64, BM, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
        return e;
    if ((e = make_tmap(&ts, f16, 2, a.s, (uint64_t)K / 32, (uint64_t)B, 16, BM, CU_TENSOR_MAP_SWIZZLE_32B)) !=
        cudaSuccess)
        return e;
    // weights as bytes [N][K/256*144]: one box = one super-block of 128 rows
    if ((e = make_tmap(&tw, u8, 1, W, (uint64_t)(K / 256) * kQ4KBlockBytes, (uint64_t)N, kQ4KBlockBytes, BN,
                       CU_TENSOR_MAP_SWIZZLE_NONE)) != cudaSuccess)
        return e;
    GemmParams p{};
    p.N = N;
    p.K = K;
    p.B = B;
    p.nb = K / 256;
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
    q4k_gemm_wide_kernel<DEBUG><<<(unsigned)grid, kThreads, smem, st>>>(ta, ts, tw, p);
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
