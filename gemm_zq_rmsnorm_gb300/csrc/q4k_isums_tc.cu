// q4k_isums_tc.cu -- the integer sub-block sums of a Q4_K x Q8_1 projection
// on the tcgen05 tensor cores, exported for inspection.
//
// For every token t, weight row n and 32-weight sub-block j this kernel
// writes I[t][n][j] = sum over the sub-block of q8 * q4, the integer dot
// product that the Q4_K x Q8_1 formulation scales by d_b * sc_j * d8 (ZINC
// docs "ROCm backend": per-block integer dot products; MIInfer README,
// "Current phase": the raw int8 GEMM that bounds the native Q4_K path).
// sm_103a has no int8 tcgen05 MMA; both operands go in as fp16 holding small
// integers (q8 with |q8| <= 127, q4 in 0..15), so every product and every
// partial sum of a sub-block (below 2^17) is exact in the fp32 accumulator and
// the export is bit-exact.  The batched projection itself runs on another
// tensor-core kernel; this one exists so the integer arithmetic of the tensor
// cores can be checked against brute force.
//
// Per sub-block the MMA (M = 128 tokens, N = 128 weight rows, K = 32 as two
// K = 16 steps) writes one of four TMEM buffers; epilogue warps read it and
// store the integers.  Warp roles (20 warps): 0 TMA producer (fp16 activation
// tiles in a six-stage ring, raw Q4_K tiles two super-blocks ahead), 1 MMA
// issuer + TMEM owner, 2-3 converters (Q4_K nibbles -> fp16 in the
// 128-byte-swizzled K-major layout, two rows per thread), 4-19 epilogue.
// Every wait is bounded.
#include <cuda.h>

#include "zq_internal.cuh"
#include "zq_tc.cuh"
#include "zq_tc_common.cuh"

namespace zq {
namespace {

constexpr int BM = 128;               // tokens per tile (TMEM lanes)
constexpr int BN = 128;               // weight rows per tile (TMEM columns)
constexpr int kAStages = 6;           // activation operand stages of K = 64 (two sub-blocks)
constexpr int kBStages = 3;           // converted weight operand stages of K = 64
constexpr int kAtomBytes = 128 * 128; // 128 rows x 64 fp16 (128 B), 128-byte swizzle
constexpr int kRawSlots = 3;          // raw Q4_K tiles in flight (super-blocks)
constexpr int kRawBytes = BN * kQ4KBlockBytes;  // 128 rows x 144 B
constexpr int kRing = 4;              // TMEM result buffers, one sub-block each
constexpr int kWarps = 20;
constexpr int kThreads = kWarps * 32;
constexpr int kConvWarp0 = 2, kConvWarps = 2;   // each converter thread owns two weight rows
constexpr int kEpiWarp0 = 4, kEpiWarps = 16;
constexpr int kEpiCols = BN / (kEpiWarps / 4);   // 32 columns per epilogue thread
constexpr uint32_t kIdesc = idesc_f16_f32(BM, BN);
constexpr uint32_t kTmemCols = 512;
static_assert(kRing * BN == (int)kTmemCols, "the result ring fills tensor memory");

struct Smem {
    // offsets from the 1024-aligned base
    static constexpr size_t a_atom(int s) { return (size_t)s * kAtomBytes; }
    static constexpr size_t b_atom(int s) { return a_atom(kAStages) + (size_t)s * kAtomBytes; }
    static constexpr size_t raw(int i) { return b_atom(kBStages) + (size_t)i * kRawBytes; }
    static constexpr size_t bars() { return raw(kRawSlots); }
    static constexpr int kNumBars = 2 * kAStages + 2 * kBStages + 2 * kRawSlots + 2 * kRing;
    static constexpr size_t tmem_slot() { return bars() + kNumBars * 8; }
    static constexpr size_t total() { return tmem_slot() + 16 + 1024; }  // + alignment slack
};
static_assert(Smem::total() <= 227 * 1024, "shared memory budget");
static_assert(kRawBytes % 1024 == 0, "raw slots keep the operand atoms 1024-byte aligned");
static_assert(Smem::total() < (1u << 18), "descriptor start addresses stay inside their 14-bit field");

struct IsumParams {
    int N, K, B, nb;
    int t_tiles;
    int32_t *isums;     // [B][N][K/32]
    unsigned int *status;
};

__global__ void __maxnreg__(96)
q4k_isums_tc_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_w,
                    const IsumParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    __shared__ volatile int abort_s;

    uint64_t *a_full = reinterpret_cast<uint64_t *>(sm + Smem::bars());
    uint64_t *a_empty = a_full + kAStages;
    uint64_t *b_full = a_empty + kAStages;
    uint64_t *b_empty = b_full + kBStages;
    uint64_t *raw_full = b_empty + kBStages;
    uint64_t *raw_empty = raw_full + kRawSlots;
    uint64_t *ring_full = raw_empty + kRawSlots;
    uint64_t *ring_empty = ring_full + kRing;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + Smem::tmem_slot());

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int t_tile = blockIdx.x % p.t_tiles;
    const int n_tile = blockIdx.x / p.t_tiles;
    const int t0 = t_tile * BM;
    const int n0 = n_tile * BN;
    const int nb = p.nb;
    const int nq = 4 * nb;   // operand stages (K = 64 each)

    if (threadIdx.x == 0) {
        for (int s = 0; s < kAStages; ++s) {
            mbar_init(&a_full[s], 1);
            mbar_init(&a_empty[s], 1);
        }
        for (int s = 0; s < kBStages; ++s) {
            mbar_init(&b_full[s], kConvWarps);
            mbar_init(&b_empty[s], 1);
        }
        for (int s = 0; s < kRawSlots; ++s) {
            mbar_init(&raw_full[s], 1);
            mbar_init(&raw_empty[s], kConvWarps);
        }
        for (int i = 0; i < kRing; ++i) {
            mbar_init(&ring_full[i], 1);
            mbar_init(&ring_empty[i], kEpiWarps);
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
            prefetch_tmap(&tmap_w);
            bool ok = true;
            int next_raw = 0;
            auto load_raw = [&](int bb) -> bool {
                const int rs = bb % kRawSlots, use = bb / kRawSlots;
                if (use > 0 && !wait_fast(&raw_empty[rs], (use - 1) & 1, &abort_s, p.status)) return false;
                mbar_arrive_expect_tx(&raw_full[rs], kRawBytes);
                tma_load_2d(sm + Smem::raw(rs), &tmap_w, kQ4KBlockBytes * bb, n0, &raw_full[rs]);
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
                if (round > 0 && !(ok = wait_fast(&a_empty[slot], (round - 1) & 1, &abort_s, p.status))) break;
                mbar_arrive_expect_tx(&a_full[slot], kAtomBytes);
                tma_load_2d(sm + Smem::a_atom(slot), &tmap_a, 256 * b + 64 * i, t0, &a_full[slot]);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t base = smem_u32(sm);
            const uint64_t a_desc0 = smem_desc(base + (uint32_t)Smem::a_atom(0), 16, 1024, kLayoutSw128);
            const uint64_t b_desc0 = smem_desc(base + (uint32_t)Smem::b_atom(0), 16, 1024, kLayoutSw128);
            constexpr uint32_t kAtom16 = kAtomBytes >> 4;
            int as = 0, bs = 0;
            uint32_t aph = 0, bph = 0, e = 0;   // e: sub-block entries issued so far
            bool ok = true;
            for (int q = 0; q < nq && ok; ++q) {
                if (!(ok = wait_fast(&a_full[as], aph, &abort_s, p.status) &&
                           wait_fast(&b_full[bs], bph, &abort_s, p.status)))
                    break;
                const uint64_t ad = a_desc0 + (uint64_t)(as * kAtom16);
                const uint64_t bd = b_desc0 + (uint64_t)(bs * kAtom16);
#pragma unroll
                for (int jj = 0; jj < 2; ++jj, ++e) {
                    const uint32_t buf = e & (kRing - 1);
                    if (e >= (uint32_t)kRing &&
                        !(ok = wait_fast(&ring_empty[buf], ((e / kRing) - 1) & 1, &abort_s, p.status)))
                        break;
                    tc_fence_after();
                    const uint32_t d_tmem = tmem + (uint32_t)BN * buf;
                    mma_f16(d_tmem, ad + (uint64_t)(jj * 4), bd + (uint64_t)(jj * 4), kIdesc, 0u);
                    mma_f16(d_tmem, ad + (uint64_t)(jj * 4 + 2), bd + (uint64_t)(jj * 4 + 2), kIdesc, 1u);
                    mma_commit(&ring_full[buf]);
                }
                if (!ok) break;
                mma_commit(&a_empty[as]);
                mma_commit(&b_empty[bs]);
                if (++as == kAStages) { as = 0; aph ^= 1u; }
                if (++bs == kBStages) { bs = 0; bph ^= 1u; }
            }
        }
    } else if (warp < kEpiWarp0) {
        // ---------------------------------------------------- converters
        // thread r converts weight rows r and r + 64 of the tile: q4 -> fp16
        const int r0 = (warp - kConvWarp0) * 32 + lane;
        const __half2 one = __float2half2_rn(1.0f), off_lo = __float2half2_rn(-1024.0f);
        const __half2 sixteenth = __float2half2_rn(0.0625f), off_hi = __float2half2_rn(-64.0f);
        for (int b = 0; b < nb; ++b) {
            const int rs = b % kRawSlots, ruse = b / kRawSlots;
            if (!warp_wait(&raw_full[rs], ruse & 1, &abort_s, p.status)) break;
            const uint8_t *rawbase = sm + Smem::raw(rs);
            bool ok = true;
            for (int i = 0; i < 4 && ok; ++i) {
                const int q = 4 * b + i;
                const int bs = q % kBStages, round = q / kBStages;
                if (round > 0 && !(ok = warp_wait(&b_empty[bs], (round - 1) & 1, &abort_s, p.status))) break;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int r = r0 + 64 * h;
                    const uint8_t *raw = rawbase + (size_t)r * kQ4KBlockBytes;
                    const uint4 n0v = *reinterpret_cast<const uint4 *>(raw + 16 + 32 * i);
                    const uint4 n1v = *reinterpret_cast<const uint4 *>(raw + 32 + 32 * i);
                    const uint32_t wv[8] = {n0v.x, n0v.y, n0v.z, n0v.w, n1v.x, n1v.y, n1v.z, n1v.w};
                    uint8_t *atom = sm + Smem::b_atom(bs) + (size_t)r * 128;
                    const int sw = r & 7;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint4 lo, hi;
                        nib4_to_h2<false>(wv[2 * c], one, off_lo, lo.x, lo.y);
                        nib4_to_h2<false>(wv[2 * c + 1], one, off_lo, lo.z, lo.w);
                        nib4_to_h2<true>(wv[2 * c], sixteenth, off_hi, hi.x, hi.y);
                        nib4_to_h2<true>(wv[2 * c + 1], sixteenth, off_hi, hi.z, hi.w);
                        *reinterpret_cast<uint4 *>(atom + ((c ^ sw) << 4)) = lo;
                        *reinterpret_cast<uint4 *>(atom + (((c + 4) ^ sw) << 4)) = hi;
                    }
                }
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&b_full[bs]);
            }
            if (!ok) break;
            __syncwarp();
            if (lane == 0) mbar_arrive(&raw_empty[rs]);
        }
    } else {
        // ---------------------------------------------------- epilogue
        const int e_w = warp - kEpiWarp0;
        const int cg = e_w >> 2;                  // column group: columns 32cg .. 32cg+31
        const int quarter = warp & 3;             // TMEM lanes 32*quarter .. +31
        const int tok = t0 + 32 * quarter + lane;
        const bool tvalid = tok < p.B;
        const uint32_t lane_base = tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(kEpiCols * cg);
        const int nsub = nb * 8;
        bool ok = true;
        for (uint32_t e = 0; e < (uint32_t)nsub && ok; ++e) {
            const uint32_t buf = e & (kRing - 1);
            if (!(ok = warp_wait(&ring_full[buf], (e / kRing) & 1, &abort_s, p.status))) break;
            tc_fence_after();
            uint32_t r[32];
            tmem_ld32(lane_base + (uint32_t)BN * buf, r);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ring_empty[buf]);
            if (tvalid) {
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const int n = n0 + kEpiCols * cg + c;
                    if (n < p.N) p.isums[((size_t)tok * p.N + n) * nsub + e] = (int32_t)__uint_as_float(r[c]);
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

size_t g_attr_bytes[64];

}  // namespace

cudaError_t launch_isums_tc(const void *W, int N, int K, zq_q8_1 a, int B, int32_t *isums, void *ws,
                            cudaStream_t st)
{
    __half *a16 = static_cast<__half *>(ws);
    cudaError_t e = launch_q8_to_f16(a.qs, a16, (size_t)B * K, st);
    if (e != cudaSuccess) return e;
    CUtensorMap ta, tw;
    if ((e = make_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a16, (uint64_t)K, (uint64_t)B, 64, BM,
                          CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
        return e;
    if ((e = make_tmap_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, W, (uint64_t)(K / 256) * kQ4KBlockBytes, (uint64_t)N,
                          kQ4KBlockBytes, BN, CU_TENSOR_MAP_SWIZZLE_NONE)) != cudaSuccess)
        return e;
    IsumParams p{};
    p.N = N;
    p.K = K;
    p.B = B;
    p.nb = K / 256;
    p.t_tiles = (B + BM - 1) / BM;
    p.isums = isums;
    p.status = device_status_word();
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    const size_t smem = Smem::total();
    if (g_attr_bytes[dev] < smem) {
        e = cudaFuncSetAttribute(q4k_isums_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        g_attr_bytes[dev] = smem;
    }
    const long long grid = (long long)p.t_tiles * ((N + BN - 1) / BN);
    q4k_isums_tc_kernel<<<(unsigned)grid, kThreads, smem, st>>>(ta, tw, p);
    return cudaGetLastError();
}

}  // namespace zq
