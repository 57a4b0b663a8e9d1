// f16_gemm_2sm.cu -- dense binary16 GEMM on the tensor cores of CTA pairs,
//   y[t][n] = sum_k x[t][k] * w[n][k]     (binary16 x and w, fp32 accumulation),
// the GEMM half of the dequantise-then-GEMM prefill (MIInfer README, "Current
// phase": Q4_K weights dequantised to 16-bit ahead of a dense GEMM, the
// pages' strongest prefill lever), measured beside the library's own
// Q4_K x Q8_1 kernel.  Each product of two binary16 values is exact in fp32;
// what separates this result from the Q4_K x Q8_1 projection is the rounding
// of the weights and of the activations to binary16 before the GEMM.
//
// Tile of a pair: 256 weight rows (128 per CTA: the MMA's M) x up to 256
// tokens (each CTA stages half: the MMA's N), K in stages of 64 (one
// 128-byte-swizzled TMA box per operand per CTA, 16 KB each; six stages).
// The kernel is persistent: pair p takes the units p, p + P, ... of
// (K split, token tile, weight tile), and the accumulator is double-buffered
// in tensor memory (2 x 256 columns), so the epilogue of one unit overlaps
// the MMAs of the next.
//
// Warps: 0 the TMA producer (lane 0; both CTAs' bytes are counted on the
// even CTA's stage barrier); 1 the MMA issuer (lane 0 of the even CTA) and
// tensor-memory owner; 2-3 idle; 4-7 the epilogue (TMEM lane quarter =
// warp % 4: 32 weight rows, all token columns).  Every wait is bounded; a
// failed wait stops both CTAs of the pair.
#include <cuda.h>

#include "zq_cluster.cuh"
#include "zq_internal.cuh"
#include "zq_pair_wait.cuh"
#include "zq_tc.cuh"
#include "zq_tc_common.cuh"

namespace zq {
namespace {

constexpr int kRows = 128;                 // weight rows per CTA (MMA M / 2)
constexpr int kTileN = 256;                // tokens per pair tile (MMA N, at most)
constexpr int kToks = kTileN / 2;          // tokens staged per CTA
constexpr int kPairM = 2 * kRows;
constexpr int kStageK = 64;                // K per stage: 128 bytes of binary16
constexpr int kStages = 6;
constexpr int kAtom = 128 * 128;           // 128 rows x 128 bytes, 128-byte swizzle
constexpr int kStageBytes = 2 * kAtom;     // weights, tokens
constexpr int kThreads = 256;
constexpr int kEpiWarp0 = 4, kEpiWarps = 4;
constexpr uint32_t kTmemCols = 2 * kTileN;   // two accumulators
static_assert(kEpiWarp0 % 4 == 0, "epilogue lane quarters follow warp % 4");
static_assert(kToks % 8 == 0 && kTileN % 16 == 0, "MMA N and the swizzle atoms' 8-row groups");

struct Smem {
    static constexpr size_t a(int s) { return (size_t)s * kStageBytes; }
    static constexpr size_t b(int s) { return a(s) + kAtom; }
    static constexpr size_t bars() { return (size_t)kStages * kStageBytes; }
    // full[6], empty[6], tfull[2], tempty[2], drain
    static constexpr int kNumBars = 2 * kStages + 5;
    static constexpr size_t tmem_slot() { return bars() + kNumBars * 8; }
    static constexpr size_t total() { return tmem_slot() + 16 + 1024; }   // + alignment slack
};
static_assert(kStageBytes % 1024 == 0, "operand atoms aligned");
static_assert(Smem::total() <= 227 * 1024, "shared memory budget");
static_assert(Smem::total() < (1u << 18), "descriptor start addresses stay inside their 14-bit field");

struct F16Params {
    int N, K, B;
    int t_tiles, m_tiles, splits, units;
    int nst;               // K stages
    size_t split_stride;   // floats between two splits' partial sums
    float *y;              // [B][N], or [splits][split_stride] partial sums
    unsigned int *status;
};

struct Unit {
    int split, t0, n, row0, s0, ns;   // n: the unit's tokens (MMA N, a multiple of 16)
};

__device__ __forceinline__ Unit unit_of(const F16Params &p, int u, uint32_t rank)
{
    Unit U;
    U.split = u % p.splits;
    const int tile = u / p.splits;
    const int t_tile = tile % p.t_tiles;
    const int m_tile = tile / p.t_tiles;
    U.t0 = t_tile * kTileN;
    U.n = min(kTileN, (p.B - U.t0 + 15) & ~15);
    U.row0 = m_tile * kPairM + kRows * (int)rank;
    U.s0 = (int)((long long)U.split * p.nst / p.splits);
    U.ns = (int)((long long)(U.split + 1) * p.nst / p.splits) - U.s0;
    return U;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
f16_gemm_2sm_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_x,
                    const F16Params p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);

    uint64_t *bm = reinterpret_cast<uint64_t *>(sm + Smem::bars());
    // full[s]: stage s landed in both CTAs (TMA bytes, even CTA's barrier);
    // empty[s]: its MMAs completed (both CTAs); tfull[i]: accumulator i is
    // complete; tempty[i]: both CTAs' epilogues have read it
    uint64_t *full = bm, *empty = bm + kStages;
    uint64_t *tfull = empty + kStages, *tempty = tfull + 2, *drain = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + Smem::tmem_slot());

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], 2 * kEpiWarps);   // the epilogue warps of both CTAs
        }
        mbar_init(drain, 1);
        s_abort = 0;
        s_status = p.status;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc_pair(tmem_slot, kTmemCols);
    tc_fence_before();
    cluster_sync();   // barriers of both CTAs initialised, tensor memory allocated in both
    tc_fence_after();
    const PairCtx ctx = pair_ctx(rank);

    if (warp == 0 && lane == 0) {
        // ---------------------------------------------------- TMA producer
        prefetch_tmap(&tmap_w);
        prefetch_tmap(&tmap_x);
        uint32_t it = 0;
        bool ok = true;
        for (int u = pair; u < p.units && ok; u += npairs) {
            const Unit U = unit_of(p, u, rank);
            // CTA r stages the unit's tokens t0 + r*n/2 .. (128 rows; the MMA
            // reads the first n/2)
            const int tok0 = U.t0 + (U.n >> 1) * (int)rank;
            for (int s = 0; s < U.ns; ++s, ++it) {
                const uint32_t slot = it % kStages, use = it / kStages;
                if (use > 0 && !(ok = pair_wait(&empty[slot], (use - 1) & 1, ctx))) break;
                const uint32_t fb = cluster_addr(smem_u32(&full[slot]), 0);
                if (rank == 0) mbar_arrive_expect_tx(&full[slot], 2u * kStageBytes);
                const int kx = kStageK * (U.s0 + s);
                tma_load_2d_pair(sm + Smem::a(slot), &tmap_w, kx, U.row0, fb);
                tma_load_2d_pair(sm + Smem::b(slot), &tmap_x, kx, tok0, fb);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA issuer
        // (the whole warp runs the loop and waits; one elected lane issues)
        if (rank == 0) {
            const uint32_t tmem = *tmem_slot;
            const uint32_t base = smem_u32(sm);
            const uint64_t a0 = smem_desc(base + (uint32_t)Smem::a(0), 16, 1024, kLayoutSw128);
            const uint64_t b0 = smem_desc(base + (uint32_t)Smem::b(0), 16, 1024, kLayoutSw128);
            constexpr uint64_t kS16 = kStageBytes >> 4;
            uint32_t it = 0;
            int j = 0;
            bool ok = true;
            for (int u = pair; u < p.units && ok; u += npairs, ++j) {
                const Unit U = unit_of(p, u, 0);
                const int buf = j & 1;
                // accumulator buf was last used by unit j - 2: both epilogues have read it
                if (j >= 2 && !(ok = __all_sync(0xffffffffu, pair_wait(&tempty[buf], ((j >> 1) - 1) & 1, ctx))))
                    break;
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(kTileN * buf);
                const uint32_t idesc = idesc_f16_f32(kPairM, (uint32_t)U.n);
                for (int s = 0; s < U.ns; ++s, ++it) {
                    const uint32_t slot = it % kStages;
                    if (!(ok = __all_sync(0xffffffffu, pair_wait(&full[slot], (it / kStages) & 1, ctx)))) break;
                    tc_fence_after();
                    const uint64_t so = (uint64_t)slot * kS16;
                    if (elect_one()) {
#pragma unroll
                        for (int kk = 0; kk < kStageK / 16; ++kk)
                            mma_f16_pair(d, a0 + so + 2 * kk, b0 + so + 2 * kk, idesc, (s | kk) != 0 ? 1u : 0u);
                        mma_commit_pair_mc(&empty[slot], 3);
                    }
                    __syncwarp();
                }
                if (ok && elect_one()) mma_commit_pair_mc(&tfull[buf], 3);
                __syncwarp();
            }
            // every MMA issued has completed before the pair tears down
            if (elect_one()) mma_commit_pair_local(drain);
            __syncwarp();
            drain_wait(drain, 0);
        }
    } else if (warp >= kEpiWarp0) {
        // ---------------------------------------------------- epilogue
        const uint32_t tmem = *tmem_slot;
        const int quarter = warp & 3;   // TMEM lanes 32*quarter .. +31
        const uint32_t tempty0 = cluster_addr(smem_u32(&tempty[0]), 0);
        int j = 0;
        for (int u = pair; u < p.units; u += npairs, ++j) {
            const Unit U = unit_of(p, u, rank);
            const int buf = j & 1;
            if (!pair_warp_wait(&tfull[buf], (uint32_t)(j >> 1) & 1, ctx)) break;
            tc_fence_after();
            const int n = U.row0 + 32 * quarter + lane;   // weight row
            const bool nvalid = n < p.N;
            float *ybase = p.y + (size_t)U.split * p.split_stride + (nvalid ? n : 0);
            const uint32_t col0 = tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(kTileN * buf);
            for (int h = 0; h < U.n; h += 32) {
                uint32_t v[32];
                tmem_ld32(col0 + (uint32_t)h, v);
                tmem_wait_ld();
                if (nvalid) {
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        const int tok = U.t0 + h + c;   // column c <-> token t0 + c
                        if (tok < p.B && h + c < U.n) ybase[(size_t)tok * p.N] = __uint_as_float(v[c]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (rank == 0)
                    mbar_arrive(&tempty[buf]);
                else
                    mbar_arrive_cluster(tempty0 + 8u * (uint32_t)buf);
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
    tc_fence_before();
    cluster_sync();   // the peer's MMAs, copies and signals are finished
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(*tmem_slot, kTmemCols);
    }
}

size_t g_attr_bytes[64];
int g_max_pairs[64];

}  // namespace

// Split-K count of the dense binary16 GEMM: the pair kernel's model (256 x
// 256 tiles over the SM pairs, waves times work per unit plus the partial
// sums' traffic), with a K stage of 64 standing in for the super-block
// unit's quarter; at least one stage per split.
int f16_gemm_splits(int B, int N, int K, int sms)
{
    int sp = choose_splits_pair(B, N, K, sms);
    const int nst = K / kStageK;
    return sp < 1 ? 1 : (sp > nst ? nst : sp);
}

size_t f16_gemm_workspace_bytes(int N, int K, int B)
{
    const int sp = f16_gemm_splits(B, N, K, num_sms());
    return sp > 1 ? (size_t)sp * split_stride(B, N) * sizeof(float) : 0;
}

cudaError_t launch_f16_gemm(const void *W16, int N, int K, const void *X16, int B, float *y, float *part,
                            cudaStream_t st)
{
    const int sms = num_sms();
    const int splits = f16_gemm_splits(B, N, K, sms);
    CUtensorMap tw, tx;
    const CUtensorMapDataType f16 = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    cudaError_t e;
    if ((e = make_tmap_2d(&tw, f16, 2, W16, (uint64_t)K, (uint64_t)N, kStageK, kRows, CU_TENSOR_MAP_SWIZZLE_128B)) !=
        cudaSuccess)
        return e;
    if ((e = make_tmap_2d(&tx, f16, 2, X16, (uint64_t)K, (uint64_t)B, kStageK, kToks, CU_TENSOR_MAP_SWIZZLE_128B)) !=
        cudaSuccess)
        return e;
    F16Params p{};
    p.N = N;
    p.K = K;
    p.B = B;
    p.t_tiles = (B + kTileN - 1) / kTileN;
    p.m_tiles = (N + kPairM - 1) / kPairM;
    p.splits = splits;
    p.units = p.t_tiles * p.m_tiles * splits;
    p.nst = K / kStageK;
    p.split_stride = split_stride(B, N);
    p.y = splits > 1 ? part : y;
    p.status = device_status_word();
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    const size_t smem = Smem::total();
    if (g_attr_bytes[dev] < smem) {
        e = cudaFuncSetAttribute(f16_gemm_2sm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        g_attr_bytes[dev] = smem;
    }
    if (g_max_pairs[dev] == 0) {
        // pairs that can be resident at once (a pair needs two SMs of one GPC)
        // (the cluster shape is the kernel's compiled one)
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(2 * (sms / 2));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = smem;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, f16_gemm_2sm_kernel, &cfg) != cudaSuccess || n < 1) {
            cudaGetLastError();
            n = sms / 2;
        }
        g_max_pairs[dev] = n;
    }
    const int pairs = p.units < g_max_pairs[dev] ? p.units : g_max_pairs[dev];
    f16_gemm_2sm_kernel<<<(unsigned)(2 * pairs), kThreads, smem, st>>>(tw, tx, p);
    if (splits == 1) return cudaGetLastError();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    return launch_splitk_reduce(part, splits, (size_t)B * N, y, st);
}

}  // namespace zq
