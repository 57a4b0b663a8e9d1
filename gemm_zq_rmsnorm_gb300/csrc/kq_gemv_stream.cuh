// kq_gemv_stream.cuh -- mat-vec of k-quant weights (Q4_K, Q5_K, Q6_K) against
// Q8_1 activations of one to a few tokens, with the weights streamed through
// shared memory by bulk (TMA) copies.  Instantiated per weight format and
// token count in q4k_gemv_stream.cu, kq_gemv_q5k.cu and kq_gemv_q6k.cu.
//
// MIInfer README, "Status": Q4_K x Q8_1 MMVQ-style projections (FFN down,
// shared gate/up; Q4_K metadata staging; packed int8 dot4; activations reused
// from on-chip memory), the Q5_K x Q8_1 MMVQ-style recurrent output
// projection (scale/min hoisting, paired nibbles) and the MMVQ-style Q6_K x
// Q8_1 LM head; "Current phase": token-batched B = 4 projections.  ZINC docs
// "ROCm backend", "Build and verify": paired Q4 projections; packed Q8
// activations for the hot Q4_K, Q5_K and Q6_K projections.
//
// The mat-vec is bound by HBM bandwidth: every weight byte is read exactly
// once.  To keep enough bytes in flight independently of register pressure,
// one persistent CTA per SM runs a producer warp that issues 1-D bulk copies
// of contiguous weight tiles (R whole rows, or a piece of one long row; rows
// are contiguous, so a tile is one copy) into a ring of large shared-memory
// stages, completing on mbarriers.  Sixteen consumer warps decode the
// super-blocks from shared memory in groups of four lanes, form the integer
// sub-block sums with dp4a against the activation rows staged once per CTA,
// apply the scales in fp32 and accumulate in registers.  Lane p of a group
// takes sub-blocks 2p and 2p+1 of a Q4_K / Q5_K block; for Q6_K it takes
// positions 8p..8p+7 of all eight 32-weight quarters, so the four lanes read
// disjoint bytes of the 210-byte block.
//
// Rows are split into segments of task groups.  When a stage holds enough
// rows, a row's segments sit in one warp, which reduces the row with shuffles
// and releases the stage on its own (warp-local rows, handed out round-robin
// across stages); long rows are split over more groups and reduced through
// shared memory after a CTA barrier.  Either way a row's summation order is a
// function of K, so every launch form gives the same y for a row.  Up to four
// matrices that read the same input (q/k/v, gate/up) share one launch.
//
// Q6_K blocks are 210 bytes, so rows and blocks are only 2-byte aligned.  The
// producer copies each tile from the 16-byte boundary below it (the bytes of
// the last tile past the last 16-byte boundary of the matrix, if any, with
// plain loads), and the consumers read the blocks with aligned 32-bit loads
// and byte permutes.
//
// With x and gamma instead of Q8_1 codes (one token) the consumers first
// compute RMSNorm and the Q8_1 packing of x themselves, in the canonical order
// of the RMSNorm+Q8_1 kernel (same bytes), straight into the shared-memory
// staging, while the producer already streams weights (one or two stages
// before the consumers' input loads are out, the rest after, so those loads
// do not queue behind the ring's copies): the normalised input never goes
// through HBM and the separate launch disappears.  The same prologue forms
// silu(gate) * up instead for the down projection.
//
// With NT > 1 the CTA stages NT tokens and every decoded weight is used for
// all of them (chunked-prefill batches of up to four tokens).
#pragma once

#include <type_traits>

#include "zq_async.cuh"
#include "zq_internal.cuh"
#include "zq_q8_1_pack.cuh"

namespace zq {
namespace stream {

enum : int { kFmtQ4K = 4, kFmtQ5K = 5, kFmtQ6K = 6 };
template <int FMT> struct Fmt;
template <> struct Fmt<kFmtQ4K> { static constexpr int kBytes = 144; };
template <> struct Fmt<kFmtQ5K> { static constexpr int kBytes = 176; };
template <> struct Fmt<kFmtQ6K> { static constexpr int kBytes = 210; };

constexpr int kConsumerWarps = 16;
constexpr int kConsumers = kConsumerWarps * 32;
static_assert((kConsumerWarps & (kConsumerWarps - 1)) == 0, "warp round-robin by mask");
constexpr int kThreads = kConsumers + 32;
constexpr int kStages = 3;
constexpr int kStageMax = 64 * 1024;
constexpr int kMaxBlk = kStageMax / 144;               // 455: blocks (>= tasks) per stage, any format
constexpr int kGroups = 8 * kConsumerWarps;            // four-lane task groups per CTA
constexpr int kSeg = 4;                                // max blocks per task
constexpr int kSmemLimit = 227 * 1024 - 1024;        // dynamic bytes: the static part pads to 1 KB
constexpr int kMaxK = 32768;                           // one row of segments per warp in the reduction
constexpr int kMaxMats = kGemvMaxMats;
constexpr size_t kBalanceMinStage = 32 * 1024;        // smallest stage the row balancing may choose
constexpr long long kBalanceMinGainPct = 8;            // ... and the least it must take off the busiest CTA

struct StreamParams {
    const uint8_t *W[kMaxMats];
    float *y[kMaxMats];
    int N[kMaxMats];
    int gstart[kMaxMats + 1];   // first row group of each matrix; gstart[nmat] = total
    int nmat;
    int K, nb;
    int ntok;             // tokens of this launch (<= NT); token t's y row is y[m] + t * N[m]
    uint32_t rowbytes;
    int R;                // rows per group
    int P;                // pieces per group (> 1 only when R == 1)
    int CB;               // blocks per piece
    int nseg;             // segments per row when rows are whole (P == 1); a function of K only
    int wl;               // warp-local rows (P == 1, nseg in 1, 2, 4, 8); a function of K only
    int total_groups;
    uint32_t stage_alloc; // bytes reserved per stage (multiple of 128)
    // input: Q8_1 planes, or (x, gamma, eps) normalised in the kernel
    const int8_t *qs;
    const __half *d;
    const __half *s;
    const float *x;
    const float *gamma;
    float eps;
    int silu;             // x, gamma are gate and up: the input is silu(gate) * up, no normalisation
    zq_q8_1 q8out;        // fused input only: codes also written here by CTA 0 (qs may be null)
    const uint8_t *pf;    // bytes for the next launch to pull into L2 once this one's are requested
    size_t pf_bytes;
    unsigned int *status;
    // Failure-path test only (zero in every product launch): waits give up
    // after wait_ns instead of the default limit, and when withhold > 0 the
    // producer of every CTA stops before issuing its stage withhold - 1, so
    // the consumers' wait for that stage must expire with no copy in flight.
    uint64_t wait_ns;
    int withhold;
};

// matrix of row group g
__device__ __forceinline__ int group_mat(const StreamParams &p, int g)
{
    int m = 0;
#pragma unroll
    for (int i = 1; i < kMaxMats; ++i) m += (i < p.nmat && g >= p.gstart[i]) ? 1 : 0;
    return m;
}

__host__ __device__ constexpr size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Activation codes are stored with 16 bytes of padding after every 64: the
// 64-byte group (Q8_1 block pair) q of super-block b starts at sb*b + 80*q,
// sb = 320.  The eight lanes of a quarter-warp (two consecutive super-blocks x
// four pairs) then start in eight different 16-byte bank groups.  The Q6_K
// lanes read 8 bytes at the same offset of four neighbouring super-blocks
// instead; a super-block stride of 352 bytes (88 words) puts those four reads
// on disjoint banks.
__host__ __device__ constexpr int act_sb(bool q6) { return q6 ? 352 : 320; }
__host__ __device__ constexpr size_t act_bytes(int K, bool q6) { return (size_t)K / 256 * act_sb(q6); }
// d8 pair and s8 pair (binary16) per Q8_1 block pair
__host__ __device__ constexpr size_t ads_bytes(int K) { return (size_t)K / 64 * 8; }

static_assert(kStages * kMaxBlk >= kMaxK / 32 + 257, "RMSNorm scratch fits in the contribution area");

struct SmemLayout {
    size_t ring, act_qs, act_ds, act_sum, contrib, bars, total;
    // sums: also stage the exact code sum of every 8 activations (int16), for
    // the Q6_K offset, in the order the Q6_K lanes read them
    __host__ __device__ SmemLayout(int K, uint32_t stage_alloc, int nt, bool sums)
    {
        ring = 0;
        act_qs = ring + (size_t)kStages * stage_alloc;
        act_ds = align_up(act_qs + (size_t)nt * act_bytes(K, sums), 16);
        act_sum = align_up(act_ds + (size_t)nt * ads_bytes(K), 16);
        contrib = align_up(act_sum + (sums ? (size_t)nt * K / 4 : 0), 16);
        bars = align_up(contrib + (size_t)nt * kStages * kMaxBlk * 4, 8);
        total = bars + (2 * kStages + 1) * 8;   // full, empty, inputs-issued
    }
};

__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c)
{
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int c)
{
    int d;
    asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Scales and mins of sub-blocks 2p and 2p+1 of a Q4_K / Q5_K header, packed
// as bytes 0 and 1 of the returned words (branch-free; p = 0..3).
__device__ __forceinline__ void pair_scales(const uint4 &hdr, int p, uint32_t &sc, uint32_t &mn)
{
    const uint32_t j = (uint32_t)(2 * p) & 3u;            // byte index within a 4-byte word
    const uint32_t sel = j | ((j + 1) << 4);                // bytes j, j+1 -> bytes 0, 1
    const uint32_t s0 = __byte_perm(hdr.y, 0, sel);         // S[j], S[j+1]
    const uint32_t s1 = __byte_perm(hdr.z, 0, sel);         // S[4+j], S[5+j]
    const uint32_t s2 = __byte_perm(hdr.w, 0, sel);         // S[8+j], S[9+j]
    const uint32_t lo_sc = s0 & 0x3F3Fu, lo_mn = s1 & 0x3F3Fu;
    const uint32_t hi_sc = (s2 & 0x0F0Fu) | ((s0 >> 2) & 0x3030u);
    const uint32_t hi_mn = ((s2 >> 4) & 0x0F0Fu) | ((s1 >> 2) & 0x3030u);
    sc = p < 2 ? lo_sc : hi_sc;
    mn = p < 2 ? lo_mn : hi_mn;
}

// Q4_K: contribution of this lane's pair of sub-blocks (2p, 2p+1; all 64
// weights) of one super-block b of a row to y.
__device__ __forceinline__ float q4k_block_part(const uint8_t *blk, int p, int b, const uint8_t *aq,
                                                const uint2 *ads)
{
    // (Q4_K staging: super-block stride 320)
    const uint4 hdr = *reinterpret_cast<const uint4 *>(blk);
    const uint4 q0 = *reinterpret_cast<const uint4 *>(blk + 16 + 32 * p);
    const uint4 q1 = *reinterpret_cast<const uint4 *>(blk + 32 + 32 * p);
    const uint8_t *ap = aq + 320 * b + 80 * p;
    const uint4 a00 = *reinterpret_cast<const uint4 *>(ap);
    const uint4 a01 = *reinterpret_cast<const uint4 *>(ap + 16);
    const uint4 a10 = *reinterpret_cast<const uint4 *>(ap + 32);
    const uint4 a11 = *reinterpret_cast<const uint4 *>(ap + 48);
    constexpr uint32_t LO = 0x0F0F0F0Fu, HI = 0xF0F0F0F0u;
    int I0 = 0, I1 = 0;
    I0 = dp4a_us(q0.x & LO, a00.x, I0);
    I1 = dp4a_us(q0.x & HI, a10.x, I1);  // high nibbles in place: 16x the true products
    I0 = dp4a_us(q0.y & LO, a00.y, I0);
    I1 = dp4a_us(q0.y & HI, a10.y, I1);
    I0 = dp4a_us(q0.z & LO, a00.z, I0);
    I1 = dp4a_us(q0.z & HI, a10.z, I1);
    I0 = dp4a_us(q0.w & LO, a00.w, I0);
    I1 = dp4a_us(q0.w & HI, a10.w, I1);
    I0 = dp4a_us(q1.x & LO, a01.x, I0);
    I1 = dp4a_us(q1.x & HI, a11.x, I1);
    I0 = dp4a_us(q1.y & LO, a01.y, I0);
    I1 = dp4a_us(q1.y & HI, a11.y, I1);
    I0 = dp4a_us(q1.z & LO, a01.z, I0);
    I1 = dp4a_us(q1.z & HI, a11.z, I1);
    I0 = dp4a_us(q1.w & LO, a01.w, I0);
    I1 = dp4a_us(q1.w & HI, a11.w, I1);
    uint32_t sc, mn;
    pair_scales(hdr, p, sc, mn);
    // exact integer scaling: |sc*I| <= 63*60960 < 2^22; I1 carries the factor 16
    const int J0 = (int)(sc & 0xFFu) * I0;
    const int J1 = (int)(sc >> 8) * (I1 >> 4);
    const float2 dd = __half22float2(*reinterpret_cast<const __half2 *>(&hdr.x));  // d, dmin
    const uint2 ds = ads[4 * b + p];
    const float2 d8 = __half22float2(*reinterpret_cast<const __half2 *>(&ds.x));
    const float2 s8 = __half22float2(*reinterpret_cast<const __half2 *>(&ds.y));
    const float main = fmaf(d8.y, (float)J1, d8.x * (float)J0);
    const float mins = fmaf((float)(mn >> 8), s8.y, (float)(mn & 0xFFu) * s8.x);
    return fmaf(dd.x, main, -dd.y * mins);
}

// ---- Q4_K with several tokens: lane p decodes sub-blocks 2p and 2p+1 once ----
struct Q4Lane {
    uint4 q0, q1;            // the 32 nibble bytes (low nibbles: sub-block 2p, high: 2p+1)
    uint32_t sc, mn;         // scales / mins of the two sub-blocks (bytes 0, 1)
    float d, dmin;
};

__device__ __forceinline__ void q4k_decode(const uint8_t *blk, int p, Q4Lane &w)
{
    const uint4 hdr = *reinterpret_cast<const uint4 *>(blk);
    w.q0 = *reinterpret_cast<const uint4 *>(blk + 16 + 32 * p);
    w.q1 = *reinterpret_cast<const uint4 *>(blk + 32 + 32 * p);
    pair_scales(hdr, p, w.sc, w.mn);
    const float2 dd = __half22float2(*reinterpret_cast<const __half2 *>(&hdr.x));
    w.d = dd.x;
    w.dmin = dd.y;
}

// the arithmetic of q4k_block_part for one token's activations
__device__ __forceinline__ float q4k_dot(const Q4Lane &w, const uint4 (&a)[4], uint2 ds)
{
    constexpr uint32_t LO = 0x0F0F0F0Fu, HI = 0xF0F0F0F0u;
    int I0 = 0, I1 = 0;
    I0 = dp4a_us(w.q0.x & LO, a[0].x, I0);
    I1 = dp4a_us(w.q0.x & HI, a[2].x, I1);
    I0 = dp4a_us(w.q0.y & LO, a[0].y, I0);
    I1 = dp4a_us(w.q0.y & HI, a[2].y, I1);
    I0 = dp4a_us(w.q0.z & LO, a[0].z, I0);
    I1 = dp4a_us(w.q0.z & HI, a[2].z, I1);
    I0 = dp4a_us(w.q0.w & LO, a[0].w, I0);
    I1 = dp4a_us(w.q0.w & HI, a[2].w, I1);
    I0 = dp4a_us(w.q1.x & LO, a[1].x, I0);
    I1 = dp4a_us(w.q1.x & HI, a[3].x, I1);
    I0 = dp4a_us(w.q1.y & LO, a[1].y, I0);
    I1 = dp4a_us(w.q1.y & HI, a[3].y, I1);
    I0 = dp4a_us(w.q1.z & LO, a[1].z, I0);
    I1 = dp4a_us(w.q1.z & HI, a[3].z, I1);
    I0 = dp4a_us(w.q1.w & LO, a[1].w, I0);
    I1 = dp4a_us(w.q1.w & HI, a[3].w, I1);
    const int J0 = (int)(w.sc & 0xFFu) * I0;
    const int J1 = (int)(w.sc >> 8) * (I1 >> 4);
    const float2 d8 = __half22float2(*reinterpret_cast<const __half2 *>(&ds.x));
    const float2 s8 = __half22float2(*reinterpret_cast<const __half2 *>(&ds.y));
    const float main = fmaf(d8.y, (float)J1, d8.x * (float)J0);
    const float mins = fmaf((float)(w.mn >> 8), s8.y, (float)(w.mn & 0xFFu) * s8.x);
    return fmaf(w.d, main, -w.dmin * mins);
}

// ---- Q5_K: lane p decodes the 5-bit quants of sub-blocks 2p and 2p+1 ----
struct Q5Lane {
    uint32_t q0[8], q1[8];   // quants 0..31, four per word, sub-blocks 2p and 2p+1
    uint32_t sc, mn;         // scales / mins of the two sub-blocks (bytes 0, 1)
    float d, dmin;
};

__device__ __forceinline__ void q5k_decode(const uint8_t *blk, int p, Q5Lane &w)
{
    const uint4 hdr = *reinterpret_cast<const uint4 *>(blk);
    const uint4 h0 = *reinterpret_cast<const uint4 *>(blk + 16);
    const uint4 h1 = *reinterpret_cast<const uint4 *>(blk + 32);
    const uint4 l0 = *reinterpret_cast<const uint4 *>(blk + 48 + 32 * p);
    const uint4 l1 = *reinterpret_cast<const uint4 *>(blk + 64 + 32 * p);
    const uint32_t qh[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
    const uint32_t ql[8] = {l0.x, l0.y, l0.z, l0.w, l1.x, l1.y, l1.z, l1.w};
    // bit 2p (2p+1) of every qh byte becomes bit 4 of the quant: a rotation
    // moves it there within its byte (bits leaving a byte are masked off)
    const uint32_t r0 = (uint32_t)(2 * p - 4) & 31u, r1 = (uint32_t)(2 * p - 3) & 31u;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t b0 = __funnelshift_r(qh[k], qh[k], r0);
        const uint32_t b1 = __funnelshift_r(qh[k], qh[k], r1);
        w.q0[k] = (ql[k] & 0x0F0F0F0Fu) | (b0 & 0x10101010u);
        w.q1[k] = ((ql[k] >> 4) & 0x0F0F0F0Fu) | (b1 & 0x10101010u);
    }
    pair_scales(hdr, p, w.sc, w.mn);
    const float2 dd = __half22float2(*reinterpret_cast<const __half2 *>(&hdr.x));
    w.d = dd.x;
    w.dmin = dd.y;
}

// a[0..1]: the 32 codes of Q8_1 block 2p, a[2..3]: block 2p+1; ds = d8 pair,
// s8 pair (binary16).
__device__ __forceinline__ float q5k_dot(const Q5Lane &w, const uint4 (&a)[4], uint2 ds)
{
    int I0 = 0, I1 = 0;
    I0 = dp4a_us(w.q0[0], a[0].x, I0);
    I0 = dp4a_us(w.q0[1], a[0].y, I0);
    I0 = dp4a_us(w.q0[2], a[0].z, I0);
    I0 = dp4a_us(w.q0[3], a[0].w, I0);
    I0 = dp4a_us(w.q0[4], a[1].x, I0);
    I0 = dp4a_us(w.q0[5], a[1].y, I0);
    I0 = dp4a_us(w.q0[6], a[1].z, I0);
    I0 = dp4a_us(w.q0[7], a[1].w, I0);
    I1 = dp4a_us(w.q1[0], a[2].x, I1);
    I1 = dp4a_us(w.q1[1], a[2].y, I1);
    I1 = dp4a_us(w.q1[2], a[2].z, I1);
    I1 = dp4a_us(w.q1[3], a[2].w, I1);
    I1 = dp4a_us(w.q1[4], a[3].x, I1);
    I1 = dp4a_us(w.q1[5], a[3].y, I1);
    I1 = dp4a_us(w.q1[6], a[3].z, I1);
    I1 = dp4a_us(w.q1[7], a[3].w, I1);
    // exact: |sc*I| <= 63*31*127*32 < 2^23
    const int J0 = (int)(w.sc & 0xFFu) * I0;
    const int J1 = (int)(w.sc >> 8) * I1;
    const float2 d8 = __half22float2(*reinterpret_cast<const __half2 *>(&ds.x));
    const float2 s8 = __half22float2(*reinterpret_cast<const __half2 *>(&ds.y));
    const float main = fmaf(d8.y, (float)J1, d8.x * (float)J0);
    const float mins = fmaf((float)(w.mn >> 8), s8.y, (float)(w.mn & 0xFFu) * s8.x);
    return fmaf(w.d, main, -w.dmin * mins);
}

// ---- Q6_K: lane p decodes positions i = 8p .. 8p+7 of all eight 32-weight
// quarters (h, c) of the block: weights k = 128h + 32c + i.  Its bytes are
// then disjoint from the other lanes' -- low bits at 64h + 32(c%2) + 8p (both
// nibbles used), top bits at 128 + 32h + 8p (all four bit pairs used) -- and
// each (h, c) chunk of 8 weights lies in one 16-weight sub-block (scale
// index 8h + 2c + p/2) and one Q8_1 block (4h + c). ----
struct Q6Lane {
    uint32_t q[8][2];   // quants 0..63 of chunk (h, c) = q[4h + c], four per word
    int sc[8];          // scale of chunk (h, c)
    float d;
};

// 32-bit word at byte offset o of a 2-byte-aligned block: aligned loads and a
// byte permute (sel = 0x3210 when the block is 4-byte aligned, else 0x5432).
__device__ __forceinline__ uint32_t ld_w32(const uint8_t *base4, int o, uint32_t sel)
{
    const uint32_t lo = *reinterpret_cast<const uint32_t *>(base4 + o);
    const uint32_t hi = *reinterpret_cast<const uint32_t *>(base4 + o + 4);
    return __byte_perm(lo, hi, sel);
}

// 8 bytes at offset o (o = 0 mod 4 relative to the block): three aligned words
__device__ __forceinline__ uint2 ld_w64(const uint8_t *base4, int o, uint32_t sel)
{
    const uint32_t w0 = *reinterpret_cast<const uint32_t *>(base4 + o);
    const uint32_t w1 = *reinterpret_cast<const uint32_t *>(base4 + o + 4);
    const uint32_t w2 = *reinterpret_cast<const uint32_t *>(base4 + o + 8);
    return make_uint2(__byte_perm(w0, w1, sel), __byte_perm(w1, w2, sel));
}

__device__ __forceinline__ void q6k_decode(const uint8_t *blk, int p, Q6Lane &w)
{
    const uint32_t mis = (uint32_t)reinterpret_cast<uintptr_t>(blk) & 2u;
    const uint8_t *base4 = blk - mis;
    const uint32_t sel = mis ? 0x5432u : 0x3210u;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint2 th = ld_w64(base4, 128 + 32 * h + 8 * p, sel);
        const uint32_t hw[2] = {th.x, th.y};
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
            const uint2 tl = ld_w64(base4, 64 * h + 32 * cc + 8 * p, sel);
            const uint32_t lw[2] = {tl.x, tl.y};
#pragma unroll
            for (int v = 0; v < 2; ++v) {
                // top-bit pair of quarter c (bits 2c, 2c+1) moved to bits 4..5
                const uint32_t t_lo = cc == 0 ? hw[v] << 4 : hw[v] << 2;   // quarter cc
                const uint32_t t_hi = cc == 0 ? hw[v] : hw[v] >> 2;        // quarter cc + 2
                w.q[4 * h + cc][v] = (lw[v] & 0x0F0F0F0Fu) | (t_lo & 0x30303030u);
                w.q[4 * h + cc + 2][v] = ((lw[v] >> 4) & 0x0F0F0F0Fu) | (t_hi & 0x30303030u);
            }
        }
    }
    // scales 8h + 2c + p/2: every second byte of the 16, from byte p/2
    const uint32_t s0 = ld_w32(base4, 192, sel), s1 = ld_w32(base4, 196, sel);
    const uint32_t s2 = ld_w32(base4, 200, sel), s3 = ld_w32(base4, 204, sel);
    const uint32_t sw[4] = {s0, s1, s2, s3};
    const int j = p >> 1;
    // byte j (chunk even) or j + 2 (chunk odd) of word (4h + c) / 2, sign-extended
#pragma unroll
    for (int q = 0; q < 8; ++q) w.sc[q] = (int)(int8_t)(uint8_t)(sw[q >> 1] >> (8 * (j + 2 * (q & 1))));
    w.d = __half2float(*reinterpret_cast<const __half *>(blk + 208));
}

__device__ __forceinline__ int sext16(uint32_t v, int half) { return half ? (int)v >> 16 : (int)(int16_t)(v & 0xFFFFu); }

// Token part of the lane's 64 weights.  ap: the super-block's codes in the
// staging (80-byte pair stride), dsp: its four (d8 pair, s8 pair) words, as:
// the exact sums of the lane's eight 8-code chunks (int16, chunk order 4h + c),
// so that sum (q - 32) * q8 = sum q * q8 - 32 * sum q8 stays an exact integer.
__device__ __forceinline__ float q6k_dot(const Q6Lane &w, const uint8_t *ap, const uint2 *dsp, uint4 as, int p)
{
    const uint32_t aw[4] = {as.x, as.y, as.z, as.w};
    float acc = 0.0f;
#pragma unroll
    for (int q = 0; q < 8; ++q) {   // Q8_1 block q = 4h + c of the super-block
        const uint2 a = *reinterpret_cast<const uint2 *>(ap + 80 * (q >> 1) + 32 * (q & 1) + 8 * p);
        int I = dp4a_us(w.q[q][0], a.x, 0);
        I = dp4a_us(w.q[q][1], a.y, I);
        I -= 32 * sext16(aw[q >> 1], q & 1);
        // exact: |sc * I| <= 128 * 8 * 32 * 127 < 2^23
        const int J = w.sc[q] * I;
        const __half2 d8 = *reinterpret_cast<const __half2 *>(&dsp[q >> 1].x);
        const float d8q = (q & 1) ? __high2float(d8) : __low2float(d8);
        acc = fmaf(d8q, (float)J, acc);
    }
    return w.d * acc;
}

template <int FMT, int NT>
__global__ void __launch_bounds__(kThreads, 1) kq_gemv_stream_kernel(const StreamParams p)
{
    constexpr int kBytes = Fmt<FMT>::kBytes;
    constexpr bool kAligned = (kBytes % 16) == 0;
    extern __shared__ __align__(1024) uint8_t smem[];
    const SmemLayout L(p.K, p.stage_alloc, NT, FMT == kFmtQ6K);
    uint8_t *ring = smem + L.ring;
    uint8_t *aq = smem + L.act_qs;
    uint2 *ads = reinterpret_cast<uint2 *>(smem + L.act_ds);
    // Q6_K: int16 sums of the 8-code chunks, lane-major: [super-block][lane p][Q8_1 block q]
    uint4 *asum = reinterpret_cast<uint4 *>(smem + L.act_sum);
    float *contrib = reinterpret_cast<float *>(smem + L.contrib);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint64_t *empty = full + kStages;
    uint64_t *xbar = empty + kStages;      // every consumer warp has issued its input loads
    __shared__ volatile int abort_s;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    constexpr int kSB = act_sb(FMT == kFmtQ6K); // staging stride of one super-block's codes
    const size_t tq = act_bytes(p.K, FMT == kFmtQ6K);   // and of one token's
    const int tds = p.K / 64;                  // and of its d8/s8 pairs (uint2 units)
    const int tas = p.K / 64;                  // and of its 8-code sums (uint4 units)
    const uint64_t wlim = p.wait_ns ? p.wait_ns : kWaitLimitNs;
    // fused input: RMSNorm prologue forms (see the consumers)
    constexpr int kGroupsPerPass = kConsumers / 4;   // blocks of 32 values per prologue pass
    constexpr int kRegPasses = 2;                    // x and gamma of up to this many passes stay in registers
    constexpr int kXPasses = 5;                      // x alone of up to this many passes stays in registers
    const bool regs = p.x != nullptr && !p.silu && (p.K >> 5) <= kRegPasses * kGroupsPerPass;
    // Stages the producer issues before the consumers' input loads are out:
    // the input (x, or the Q8_1 rows) is read after the programmatic-launch
    // wait, and a request issued behind the ring's first copies waits for
    // them.  One stage when the prologue reads its input once; two when it
    // loads again after its first loads (gamma of the later passes of a long
    // row, or x and gamma pass by pass), so that its second round trip has
    // fewer copies ahead of it.
    const uint32_t early = (p.x == nullptr || regs) ? 1u : 2u;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        mbar_init(xbar, kConsumerWarps);
        abort_s = 0;
        fence_mbar_init();
        pdl_launch_dependents();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t policy = l2_evict_first_policy();
            uint32_t it = 0;
            for (int g = blockIdx.x; g < p.total_groups; g += gridDim.x) {
                const int mat = group_mat(p, g);
                const int row0 = (g - p.gstart[mat]) * p.R;
                const int rows = min(p.R, p.N[mat] - row0);
                for (int pc = 0; pc < p.P; ++pc, ++it) {
                    const uint32_t slot = it % kStages, round = it / kStages;
                    if (p.withhold > 0 && it == (uint32_t)(p.withhold - 1)) return;
                    if (it == early && !mbar_wait_for(xbar, 0, p.status, wlim)) return;
                    if (round > 0 && !mbar_wait_for(&empty[slot], (round & 1) ^ 1, p.status, wlim)) return;
                    const size_t bytes = (p.P == 1) ? (size_t)rows * p.rowbytes
                                                    : (size_t)min(p.CB, p.nb - pc * p.CB) * kBytes;
                    const size_t start = (size_t)row0 * p.rowbytes + (size_t)pc * p.CB * kBytes;
                    uint8_t *dst = ring + (size_t)slot * p.stage_alloc;
                    if (kAligned) {
                        mbar_arrive_expect_tx(&full[slot], (uint32_t)bytes);
                        bulk_g2s_hint(dst, p.W[mat] + start, (uint32_t)bytes, &full[slot], policy);
                    } else {
                        // copy from the 16-byte boundary below the tile; bytes past
                        // the matrix's last 16-byte boundary go by plain loads
                        const size_t end = start + bytes;
                        const size_t total = (size_t)p.N[mat] * p.rowbytes;
                        const size_t lo = start & ~(size_t)15;
                        const size_t hi = min((end + 15) & ~(size_t)15, total & ~(size_t)15);
                        for (size_t o = hi; o < end; ++o) dst[o - lo] = __ldg(p.W[mat] + o);
                        if (end > hi) fence_async_smem();
                        mbar_arrive_expect_tx(&full[slot], (uint32_t)(hi - lo));
                        bulk_g2s_hint(dst, p.W[mat] + lo, (uint32_t)(hi - lo), &full[slot], policy);
                    }
                }
            }
            // every weight byte of this CTA is requested: while the consumers
            // finish, warm L2 with this CTA's share of the bytes the next
            // launch will stream
            if (p.pf != nullptr) {
                const size_t share = ((p.pf_bytes + gridDim.x - 1) / gridDim.x + 15) & ~(size_t)15;
                const size_t b0 = (size_t)blockIdx.x * share;
                const size_t b1 = min(b0 + share, p.pf_bytes & ~(size_t)15);
                for (size_t o = b0; o < b1; o += 65536)
                    bulk_prefetch_l2(p.pf + o, (uint32_t)min((size_t)65536, b1 - o));
            }
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    // The producer streams weights (written by no kernel) from the start (its
    // first one or two stages; the rest once every consumer warp has issued
    // its input loads); the activations may come from the previous kernel on
    // the stream, and y may still be read by it: wait for that kernel before
    // touching either.  The
    // RMSNorm weight gamma is a weight too: when the input is short enough to
    // stay in registers, it is loaded before the wait.
    const int grp = tid >> 2, sub = tid & 3;
    const bool xregs = p.x != nullptr && !p.silu && !regs && (p.K >> 5) <= kXPasses * kGroupsPerPass;
    float4 gr[kRegPasses][2];
    if (regs || xregs) {
#pragma unroll
        for (int u = 0; u < kRegPasses; ++u) {
            const int b = kGroupsPerPass * u + grp;
            const float4 *pg = reinterpret_cast<const float4 *>(p.gamma + 32 * b) + 2 * sub;
            gr[u][0] = b < (p.K >> 5) ? __ldg(pg) : make_float4(0.f, 0.f, 0.f, 0.f);
            gr[u][1] = b < (p.K >> 5) ? __ldg(pg + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    pdl_wait();
    // this warp's input loads are issued: the producer may stream the rest
    auto inputs_out = [&]() {
        __syncwarp();
        if (lane == 0) mbar_arrive(xbar);
    };
    if (p.x == nullptr) {
        inputs_out();
        // stage the activation rows: codes with the 80-byte group stride,
        // scales and sums as they are (pairs of binary16 per 32-bit word)
        for (int t = 0; t < p.ntok; ++t) {
            const uint4 *gq = reinterpret_cast<const uint4 *>(p.qs + (size_t)t * p.K);
            uint8_t *aqt = aq + t * tq;
            int16_t *at = reinterpret_cast<int16_t *>(asum + t * tas);
            for (int c = tid; c < p.K / 16; c += kConsumers) {
                const uint4 v = __ldg(gq + c);
                *reinterpret_cast<uint4 *>(aqt + kSB * (c >> 4) + 80 * ((c >> 2) & 3) + 16 * (c & 3)) = v;
                if constexpr (FMT == kFmtQ6K) {
                    // 8-code chunks 2c and 2c+1: super-block k8 / 32, lane k8 % 4, Q8_1 block (k8 % 32) / 4
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int k8 = 2 * c + e;
                        const int sum = dp4a_ss(e ? v.w : v.y, 0x01010101u, dp4a_ss(e ? v.z : v.x, 0x01010101u, 0));
                        at[((k8 >> 5) * 4 + (k8 & 3)) * 8 + ((k8 & 31) >> 2)] = (int16_t)sum;
                    }
                }
            }
            const uint32_t *gd = reinterpret_cast<const uint32_t *>(p.d + (size_t)t * (p.K / 32));
            const uint32_t *gs = reinterpret_cast<const uint32_t *>(p.s + (size_t)t * (p.K / 32));
            for (int c = tid; c < p.K / 64; c += kConsumers)
                ads[t * tds + c] = make_uint2(__ldg(gd + c), __ldg(gs + c));
        }
    } else {
        // RMSNorm + Q8_1 of x in the canonical order (per-block fma chains,
        // 256 slots in increasing block order, pairwise tree), packed into
        // the staging; scratch in the (still unused) contribution area.
        // Four lanes share a 32-value block, each holding eight consecutive
        // values, so every load instruction of a warp reads 1 KB of
        // consecutive bytes; the block's fma chain runs through the four lanes
        // in order (shuffles), and amax and the code sum are exact group
        // reductions.  (One token: the host launches this form with NT = 1.)
        const int nblk = p.K >> 5;
        float *part = contrib;                // [nblk]
        float *slot = contrib + kMaxK / 32;   // [256] and r
        constexpr int kUnroll = 3;            // passes with loads in flight together
        // sum of squares of this group's block: an fma chain through the four lanes in order
        auto chain = [&](const float4 (&xv)[2]) {
            float pr = 0.0f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (sub == j) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        pr = __fmaf_rn(xv[h].x, xv[h].x, pr);
                        pr = __fmaf_rn(xv[h].y, xv[h].y, pr);
                        pr = __fmaf_rn(xv[h].z, xv[h].z, pr);
                        pr = __fmaf_rn(xv[h].w, xv[h].w, pr);
                    }
                }
                pr = __shfl_sync(0xffffffffu, pr, (lane & ~3) | j);
            }
            return pr;
        };
        float r = 1.0f;
        // the 256 slots and the pairwise tree over the block sums: r.  The
        // tree's levels 128, 64 and 32 run in warp 0 from the slots in shared
        // memory, in the tree's own association (lane l: level 128 pairs
        // slots l + 32 j and l + 32 j + 128, level 64 pairs the results for j
        // and j + 2, level 32 those for j = 0 and 1), then levels 16 .. 1 by
        // shuffles: the same additions with three barriers instead of seven
        // (two for rows of at most 256 blocks).
        // (Rows of at most 256 blocks: a slot holds at most one block, and
        // +0 + p = p exactly, so warp 0 reads the block sums directly.)
        const bool one_per_slot = nblk <= 256;
        auto tree = [&]() {
            named_bar(1, kConsumers);
            if (!one_per_slot) {
                if (tid < 256) {
                    float v = 0.0f;
                    for (int b = tid; b < nblk; b += 256) v = __fadd_rn(v, part[b]);
                    slot[tid] = v;
                }
                named_bar(1, kConsumers);
            }
            if (warp == 0) {
                float sl[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int t = lane + 32 * j;
                    sl[j] = one_per_slot ? (t < nblk ? part[t] : 0.0f) : slot[t];
                }
                const float a0 = __fadd_rn(sl[0], sl[4]), a1 = __fadd_rn(sl[1], sl[5]);
                const float a2 = __fadd_rn(sl[2], sl[6]), a3 = __fadd_rn(sl[3], sl[7]);
                float v = __fadd_rn(__fadd_rn(a0, a2), __fadd_rn(a1, a3));
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) v = __fadd_rn(v, __shfl_down_sync(0xffffffffu, v, off));
                if (lane == 0) slot[256] = rms_scale(v, p.K, p.eps);
            }
            named_bar(1, kConsumers);
            r = slot[256];
        };
        __half *ads16 = reinterpret_cast<__half *>(ads);
        const bool out = blockIdx.x == 0 && p.q8out.qs != nullptr;
        // normalise (or form silu(gate) * up for) block b and pack it into the staging
        auto pack = [&](int b, const float4 (&xv)[2], const float4 (&gv)[2]) {
            float xh[8];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                if (p.silu) {
                    xh[4 * h + 0] = silu_mul(xv[h].x, gv[h].x);
                    xh[4 * h + 1] = silu_mul(xv[h].y, gv[h].y);
                    xh[4 * h + 2] = silu_mul(xv[h].z, gv[h].z);
                    xh[4 * h + 3] = silu_mul(xv[h].w, gv[h].w);
                } else {
                    xh[4 * h + 0] = __fmul_rn(__fmul_rn(xv[h].x, r), gv[h].x);
                    xh[4 * h + 1] = __fmul_rn(__fmul_rn(xv[h].y, r), gv[h].y);
                    xh[4 * h + 2] = __fmul_rn(__fmul_rn(xv[h].z, r), gv[h].z);
                    xh[4 * h + 3] = __fmul_rn(__fmul_rn(xv[h].w, r), gv[h].w);
                }
            }
            float amax = 0.0f;
#pragma unroll
            for (int c = 0; c < 8; ++c) amax = fmaxf(amax, fabsf(xh[c]));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
            const float d = __fdiv_rn(amax, 127.0f);
            const float id = (d != 0.0f) ? __fdiv_rn(1.0f, d) : 0.0f;
            uint32_t word[2] = {0u, 0u};
            int qsum = 0;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                float q = roundf(__fmul_rn(xh[c], id));
                q = fminf(fmaxf(q, -127.0f), 127.0f);
                const int qi = (int)q;
                qsum += qi;
                word[c >> 2] |= ((uint32_t)(qi & 0xFF)) << (8 * (c & 3));
            }
            if constexpr (FMT == kFmtQ6K) {
                // this lane's 8 codes are chunk k8 = 4b + sub
                if (b < nblk) reinterpret_cast<int16_t *>(asum)[((b >> 3) * 4 + sub) * 8 + (b & 7)] = (int16_t)qsum;
            }
            qsum += __shfl_xor_sync(0xffffffffu, qsum, 1);
            qsum += __shfl_xor_sync(0xffffffffu, qsum, 2);
            if (b < nblk) {
                *reinterpret_cast<uint2 *>(aq + kSB * (b >> 3) + 80 * ((b >> 1) & 3) + 32 * (b & 1) + 8 * sub) =
                    make_uint2(word[0], word[1]);
                const __half dh = __float2half_rn(d), sh = __float2half_rn(__fmul_rn(d, (float)qsum));
                if (sub == 0) {
                    ads16[4 * (b >> 1) + (b & 1)] = dh;
                    ads16[4 * (b >> 1) + 2 + (b & 1)] = sh;
                }
                if (out) {
                    reinterpret_cast<uint2 *>(p.q8out.qs + 32 * b)[sub] = make_uint2(word[0], word[1]);
                    if (sub == 0) {
                        reinterpret_cast<__half *>(p.q8out.d)[b] = dh;
                        reinterpret_cast<__half *>(p.q8out.s)[b] = sh;
                    }
                }
            }
        };
        if (regs) {
            // short input: x read once into registers (gamma is already there),
            // one round trip to memory after the wait instead of two.  One pass
            // or two (a compile-time count, so both passes of a two-pass row run
            // without a branch between them and their chains interleave, and a
            // one-pass row, as in small models, pays for no pass of zeros).
            auto short_prologue = [&](auto npc) {
                constexpr int NP = decltype(npc)::value;
                float4 xr[NP][2];
#pragma unroll
                for (int u = 0; u < NP; ++u) {
                    const int b = kGroupsPerPass * u + grp;
                    const float4 *px = reinterpret_cast<const float4 *>(p.x + 32 * b) + 2 * sub;
                    xr[u][0] = b < nblk ? __ldg(px) : make_float4(0.f, 0.f, 0.f, 0.f);
                    xr[u][1] = b < nblk ? __ldg(px + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
                inputs_out();
#pragma unroll
                for (int u = 0; u < NP; ++u) {
                    const int b = kGroupsPerPass * u + grp;
                    const float pr = chain(xr[u]);
                    if (sub == 0 && b < nblk) part[b] = pr;
                }
                tree();
#pragma unroll
                for (int u = 0; u < NP; ++u) pack(kGroupsPerPass * u + grp, xr[u], gr[u]);
            };
            static_assert(kRegPasses == 2, "one-pass and two-pass forms");
            if (nblk <= kGroupsPerPass)   // CTA-uniform
                short_prologue(std::integral_constant<int, 1>{});
            else
                short_prologue(std::integral_constant<int, 2>{});
        } else if (xregs) {
            // medium input (K <= 20480): x read once into registers; gamma of
            // the first two passes is already there, the rest is loaded while
            // those are packed -- two round trips after the wait instead of
            // four.  Every pass runs (a block past the row is zeros and stores
            // nothing), so the passes' dependency chains interleave.
            float4 xr[kXPasses][2];
#pragma unroll
            for (int u = 0; u < kXPasses; ++u) {
                const int b = kGroupsPerPass * u + grp;
                const float4 *px = reinterpret_cast<const float4 *>(p.x + 32 * b) + 2 * sub;
                xr[u][0] = b < nblk ? __ldg(px) : make_float4(0.f, 0.f, 0.f, 0.f);
                xr[u][1] = b < nblk ? __ldg(px + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            inputs_out();
#pragma unroll
            for (int u = 0; u < kXPasses; ++u) {
                const int b = kGroupsPerPass * u + grp;
                const float pr = chain(xr[u]);
                if (sub == 0 && b < nblk) part[b] = pr;
            }
            tree();
            // the first two passes first, so their registers are free before
            // the rest of gamma arrives
#pragma unroll
            for (int u = 0; u < kRegPasses; ++u) pack(kGroupsPerPass * u + grp, xr[u], gr[u]);
            float4 g2[kXPasses - kRegPasses][2];
#pragma unroll
            for (int u = 0; u < kXPasses - kRegPasses; ++u) {
                const int b = kGroupsPerPass * (u + kRegPasses) + grp;
                const float4 *pg = reinterpret_cast<const float4 *>(p.gamma + 32 * b) + 2 * sub;
                g2[u][0] = b < nblk ? __ldg(pg) : make_float4(0.f, 0.f, 0.f, 0.f);
                g2[u][1] = b < nblk ? __ldg(pg + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < kXPasses - kRegPasses; ++u)
                pack(kGroupsPerPass * (u + kRegPasses) + grp, xr[u + kRegPasses], g2[u]);
        } else {
            inputs_out();
            for (int base = 0; base < (p.silu ? 0 : nblk); base += kGroupsPerPass * kUnroll) {
                float4 xv[kUnroll][2];
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    if (base + kGroupsPerPass * u >= nblk) break;   // CTA-uniform
                    const int b = base + kGroupsPerPass * u + grp;
                    const float4 *px = reinterpret_cast<const float4 *>(p.x + 32 * b) + 2 * sub;
                    xv[u][0] = b < nblk ? __ldg(px) : make_float4(0.f, 0.f, 0.f, 0.f);
                    xv[u][1] = b < nblk ? __ldg(px + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    if (base + kGroupsPerPass * u >= nblk) break;
                    const int b = base + kGroupsPerPass * u + grp;
                    const float pr = chain(xv[u]);
                    if (sub == 0 && b < nblk) part[b] = pr;
                }
            }
            if (!p.silu) tree();
            for (int base = 0; base < nblk; base += kGroupsPerPass * kUnroll) {
                float4 xv[kUnroll][2], gv[kUnroll][2];
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    if (base + kGroupsPerPass * u >= nblk) break;
                    const int b = base + kGroupsPerPass * u + grp;
                    const bool in = b < nblk;
                    const float4 *px = reinterpret_cast<const float4 *>(p.x + 32 * b) + 2 * sub;
                    const float4 *pg = reinterpret_cast<const float4 *>(p.gamma + 32 * b) + 2 * sub;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        xv[u][h] = in ? __ldg(px + h) : make_float4(0.f, 0.f, 0.f, 0.f);
                        gv[u][h] = in ? __ldg(pg + h) : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    if (base + kGroupsPerPass * u >= nblk) break;
                    pack(base + kGroupsPerPass * u + grp, xv[u], gv[u]);
                }
            }
        }
    }
    named_bar(1, kConsumers);

    // Work of a stage: each row's blocks are split into nseg strided segments
    // (segment s takes blocks s, s + nseg, ...); a task is one (row, segment)
    // and runs on one group of four lanes, which accumulates in registers.
    // Neighbouring groups take neighbouring segments, i.e. neighbouring blocks,
    // so their shared-memory reads fall in different bank groups.
    const int G = warp * 8 + (lane >> 2);   // task group, 128 per CTA
    const int pp = lane & 3;                // Q8_1 block pair 2pp, 2pp+1
    const unsigned gmask = 0xFu << (4 * (lane >> 2));
    // warp-local rows: nseg (a power of two, 1..8) task groups per row, so
    // 8 / nseg = 2^(3 - wl_lg) rows per slot of eight groups; this lane's
    // segment and row within a slot (launch constants, hoisted out of the
    // stage loop)
    const int wl_lg = p.wl ? __ffs(p.nseg) - 1 : 0;
    const int wl_sg = (lane >> 2) & (p.nseg - 1), wl_sr = (lane >> 2) >> wl_lg;
    uint32_t it = 0;
    uint32_t rr = 0;                        // warp-local rows: slots handed out so far
    for (int g = blockIdx.x; g < p.total_groups; g += gridDim.x) {
        const int mat = group_mat(p, g);
        const int row0 = (g - p.gstart[mat]) * p.R;
        const int rows = min(p.R, p.N[mat] - row0);
        float *yv = p.y[mat];
        const size_t ytok = (size_t)p.N[mat];
        float row_acc[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) row_acc[t] = 0.0f;
        for (int pc = 0; pc < p.P; ++pc, ++it) {
            const uint32_t slot = it % kStages, round = it / kStages;
            // every lane observes the completed phase itself (acquire) before
            // reading the stage: one warp-wide wait, whose lanes see the same
            // barrier state (a lane-0 poll followed by a shuffle and a second
            // wait cost more per stage: 0.3 us on the small launches)
            if (p.wl && abort_s) return;
            const bool ok = mbar_wait_for(&full[slot], round & 1, p.status, wlim);
            if (!ok) abort_s = 1;
            // the tile starts (start mod 16) bytes into the stage
            const size_t start = (size_t)row0 * p.rowbytes + (size_t)pc * p.CB * kBytes;
            const uint8_t *stage = ring + (size_t)slot * p.stage_alloc + (kAligned ? 0 : (start & 15));
            float *cb = contrib + slot * kMaxBlk;
            // blocks per row in this stage and where they start in the row
            const int rowblk = (p.P == 1) ? p.nb : min(p.CB, p.nb - pc * p.CB);
            const int bbase = pc * p.CB;
            const int nrows = (p.P == 1) ? rows : 1;
            const int nseg = (p.P == 1) ? p.nseg : (rowblk + kSeg - 1) / kSeg;
            const int ntask = nrows * nseg;
            // partial sums of this lane's 64 weights of block lb of a row, per token
            auto block = [&](const uint8_t *rowp, int lb, float (&out)[NT]) {
                const uint8_t *blk = rowp + (size_t)lb * kBytes;
                const int b = bbase + lb;        // super-block index in the row
                if constexpr (FMT == kFmtQ4K && NT == 1) {
                    out[0] = q4k_block_part(blk, pp, b, aq, ads);
                } else {
                    typename std::conditional<FMT == kFmtQ4K, Q4Lane,
                        typename std::conditional<FMT == kFmtQ5K, Q5Lane, Q6Lane>::type>::type w;
                    if constexpr (FMT == kFmtQ4K) q4k_decode(blk, pp, w);
                    else if constexpr (FMT == kFmtQ5K) q5k_decode(blk, pp, w);
                    else q6k_decode(blk, pp, w);
#pragma unroll
                    for (int tk = 0; tk < NT; ++tk) {
                        if (tk < p.ntok) {
                            if constexpr (FMT != kFmtQ6K) {
                                const uint8_t *ap = aq + tk * tq + kSB * b + 80 * pp;
                                const uint4 a[4] = {*reinterpret_cast<const uint4 *>(ap),
                                                    *reinterpret_cast<const uint4 *>(ap + 16),
                                                    *reinterpret_cast<const uint4 *>(ap + 32),
                                                    *reinterpret_cast<const uint4 *>(ap + 48)};
                                if constexpr (FMT == kFmtQ4K) out[tk] = q4k_dot(w, a, ads[tk * tds + 4 * b + pp]);
                                else out[tk] = q5k_dot(w, a, ads[tk * tds + 4 * b + pp]);
                            } else {
                                out[tk] = q6k_dot(w, aq + tk * tq + kSB * b, ads + tk * tds + 4 * b,
                                                  asum[tk * tas + 4 * b + pp], pp);
                            }
                        } else {
                            out[tk] = 0.0f;
                        }
                    }
                }
            };
            if (p.wl && p.P == 1) {
                // Warp-local rows: the nseg (1, 2, 4 or 8) task groups of a row
                // sit in one warp, which reduces the row with shuffles and writes
                // y; each warp releases the stage on its own.  Slots of 8/nseg
                // rows go to the warps round-robin, continuing across stages.
                if (!ok) return;
                const int nslots = (nrows + (8 >> wl_lg) - 1) >> (3 - wl_lg);
                const int sg = wl_sg;
                const int s0 = (int)((uint32_t)(warp - (int)rr) & (kConsumerWarps - 1));
                for (int sl = s0; sl < nslots; sl += kConsumerWarps) {
                    const int r = (sl << (3 - wl_lg)) + wl_sr;   // row within the stage
                    const bool live = r < nrows;
                    const uint8_t *rowp = stage + (size_t)(live ? r : 0) * rowblk * kBytes;
                    float c[NT];
#pragma unroll
                    for (int tk = 0; tk < NT; ++tk) c[tk] = 0.0f;
                    // blocks sg, sg + nseg, ... of the row, summed in order: four at
                    // a time with no condition between them (so their loads are in
                    // flight together) while four remain, then one at a time
                    int lb = sg;
                    for (; live && lb + (kSeg - 1) * nseg < rowblk; lb += kSeg * nseg) {
                        float part[kSeg][NT];
#pragma unroll
                        for (int i = 0; i < kSeg; ++i) block(rowp, lb + i * nseg, part[i]);
#pragma unroll
                        for (int i = 0; i < kSeg; ++i)
#pragma unroll
                            for (int tk = 0; tk < NT; ++tk) c[tk] += part[i][tk];
                    }
                    for (; live && lb < rowblk; lb += nseg) {
                        float part[NT];
                        block(rowp, lb, part);
#pragma unroll
                        for (int tk = 0; tk < NT; ++tk) c[tk] += part[tk];
                    }
#pragma unroll
                    for (int tk = 0; tk < NT; ++tk) {
                        float v = c[tk];
                        v += __shfl_xor_sync(0xffffffffu, v, 1);
                        v += __shfl_xor_sync(0xffffffffu, v, 2);
                        for (int off = 4; off < 4 * nseg; off <<= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
                        if (live && (lane & (4 * nseg - 1)) == 0 && tk < p.ntok) yv[tk * ytok + row0 + r] = v;
                    }
                }
                rr += (uint32_t)nslots;
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[slot]);
                continue;
            }
            if (ok) {
                for (int t = G; t < ntask; t += kGroups) {
                    const int r = t / nseg;
                    const int sg = t - r * nseg;
                    const uint8_t *rowp = stage + (size_t)r * rowblk * kBytes;
                    float c[NT];
                    if (nseg == rowblk) {
                        // short rows: one block per task
                        block(rowp, sg, c);
                    } else {
                        // all of the segment's blocks are read unconditionally (a
                        // block past the row end re-reads the first one and is
                        // dropped), so their shared-memory loads can all be in
                        // flight together; the sum keeps the segment order
                        float part[kSeg][NT];
#pragma unroll
                        for (int i = 0; i < kSeg; ++i) {
                            const int lb0 = sg + i * nseg;   // block within this stage's row
                            block(rowp, lb0 < rowblk ? lb0 : sg, part[i]);
                        }
#pragma unroll
                        for (int tk = 0; tk < NT; ++tk) {
                            c[tk] = 0.0f;
#pragma unroll
                            for (int i = 0; i < kSeg; ++i)
                                if (sg + i * nseg < rowblk) c[tk] += part[i][tk];
                        }
                    }
#pragma unroll
                    for (int tk = 0; tk < NT; ++tk) {
                        float v = c[tk];
                        v += __shfl_xor_sync(gmask, v, 1);
                        v += __shfl_xor_sync(gmask, v, 2);
                        if (pp == 0) cb[(size_t)tk * kStages * kMaxBlk + t] = v;
                    }
                }
            }
            named_bar(1, kConsumers);
            if (abort_s) return;
            if (lane == 0) mbar_arrive(&empty[slot]);
            if (p.P == 1) {
                for (int r = warp; r < rows; r += kConsumerWarps) {
                    for (int tk = 0; tk < p.ntok; ++tk) {
                        const float *cbt = cb + (size_t)tk * kStages * kMaxBlk;
                        float v = lane < nseg ? cbt[r * nseg + lane] : 0.0f;
#pragma unroll
                        for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
                        if (lane == 0) yv[tk * ytok + row0 + r] = v;
                    }
                }
            } else if (warp == 0) {
#pragma unroll
                for (int tk = 0; tk < NT; ++tk) {
                    if (tk >= p.ntok) break;
                    const float *cbt = cb + (size_t)tk * kStages * kMaxBlk;
                    float v = 0.0f;
                    for (int q = lane; q < nseg; q += 32) v += cbt[q];
#pragma unroll
                    for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
                    row_acc[tk] += v;
                    if (pc == p.P - 1 && lane == 0) yv[tk * ytok + row0] = row_acc[tk];
                }
            }
        }
    }
}

// The launch plan -- rows per stage, pieces, segments, warp-local mode, stage
// size -- for K columns, totalN rows in all and sms CTAs: a pure host
// computation (checked on the CPU through zq_debug_stream_plan).  Returns false
// when the activation staging leaves no room for the stages.
template <int FMT, int NT>
bool plan_stream(StreamParams &p, int K, long long totalN, int sms)
{
    constexpr int kBytes = Fmt<FMT>::kBytes;
    // an unaligned tile is copied from up to 14 bytes below its start to up to
    // 14 bytes past its end; the last block's aligned loads read 2 bytes past it
    constexpr uint32_t kSlack = (kBytes % 16) ? 32 : 0;
    p.K = K;
    p.nb = K / 256;
    p.rowbytes = (uint32_t)p.nb * kBytes;
    // stage size: as large as shared memory allows (<= 64 KB), but small
    // enough that every CTA gets >= 3 stages of work
    const size_t fixed = SmemLayout(K, 0, NT, FMT == kFmtQ6K).total;
    if (fixed + (size_t)kStages * align_up(kBytes + kSlack, 128) > (size_t)kSmemLimit) return false;
    size_t cap = (kSmemLimit - fixed) / kStages / 128 * 128;
    cap = cap > (size_t)kStageMax ? (size_t)kStageMax : cap;
    const double total = (double)totalN * p.rowbytes;
    size_t target = (size_t)(total / sms / 3);
    target = target < 4096 ? 4096 : (target > cap ? cap : target);
    // A row is split into pieces only when it does not fit in a stage at all,
    // so a row's summation order depends on K alone, not on which other
    // matrices share the launch.
    // Segments per row.  Warp-local rows: nseg of 4, 8, 2 or 1 task groups in
    // one warp, the choice that splits the row's blocks most evenly among
    // those for which a full stage holds rows for five or more warps (so the
    // three stages in flight keep the sixteen warps busy).  Otherwise (long
    // rows) segments of up to kSeg blocks reduced through shared memory.  Both
    // depend on K (and the format and token count) only, so a row's summation
    // order does not depend on the other matrices of a launch.
    const long long rcap = p.rowbytes + kSlack <= cap ? (long long)((cap - kSlack) / p.rowbytes) : 0;
    int ns_wl = 0;
    double best_u = -1.0;
    for (int ns : {4, 8, 2, 1}) {
        if (rcap * ns < 40) continue;
        const double u = (double)p.nb / (double)(ns * ((p.nb + ns - 1) / ns));
        if (u > best_u + 1e-12) {
            best_u = u;
            ns_wl = ns;
        }
    }
    p.wl = ns_wl > 0 ? 1 : 0;
    p.nseg = p.wl ? ns_wl : (p.nb <= 8 ? p.nb : (p.nb + kSeg - 1) / kSeg);
    if (p.rowbytes + kSlack <= cap) {
        const int rmax = p.rowbytes + kSlack <= target ? (int)((target - kSlack) / p.rowbytes) : 1;
        // rows per stage: the most rows per round of task groups (a stage of
        // R rows takes ceil(R*nseg/128) rounds), among R in [rmax/2, rmax];
        // warp-local rows are balanced across stages, any R will do
        p.R = rmax;
        for (int r = rmax; !p.wl && r >= (rmax + 1) / 2; --r) {
            const long long rounds_r = ((long long)r * p.nseg + kGroups - 1) / kGroups;
            const long long rounds_R = ((long long)p.R * p.nseg + kGroups - 1) / kGroups;
            if ((long long)r * rounds_R > (long long)p.R * rounds_r) p.R = r;
        }
        // warp-local rows: the row groups go to the CTAs round-robin, so pick
        // the R that leaves the fewest rows on the busiest CTA (the launch
        // ends with it), among stages of at least half the largest and of
        // 32 KB or more, when that takes 8 % or more off it (smaller stages
        // cost more per byte than a small gain in balance); a row's
        // summation order does not depend on R
        if (p.wl) {
            auto load = [&](int r) { return ((totalN + r - 1) / r + sms - 1) / sms * r; };
            const long long full = load(rmax);
            long long best = full;
            int rb = rmax;
            const int rlo = max((rmax + 1) / 2, (int)((kBalanceMinStage + p.rowbytes - 1) / p.rowbytes));
            for (int r = rmax - 1; r >= rlo; --r)
                if (load(r) < best) {
                    best = load(r);
                    rb = r;
                }
            // (measured: smaller stages pay off only for a clear gain)
            if (best * 100 <= full * (100 - kBalanceMinGainPct)) p.R = rb;
        }
        p.P = 1;
        p.CB = p.nb;
        p.stage_alloc = (uint32_t)align_up((size_t)p.R * p.rowbytes + kSlack, 128);
    } else {
        p.R = 1;
        p.CB = (int)((cap - kSlack) / kBytes);
        if (p.CB < 1) p.CB = 1;
        p.P = (p.nb + p.CB - 1) / p.CB;
        p.stage_alloc = (uint32_t)align_up((size_t)p.CB * kBytes + kSlack, 128);
    }
    return true;
}

// Bytes of dynamic shared memory a plan uses.
template <int FMT, int NT>
size_t plan_smem(const StreamParams &p)
{
    return SmemLayout(p.K, p.stage_alloc, NT, FMT == kFmtQ6K).total;
}

// Host side: tile the job, size the stages and launch.  Returns
// cudaErrorInvalidValue when the activation staging does not fit.
// ctas > 0 plans and launches for that many CTAs instead of one per SM.
template <int FMT, int NT>
cudaError_t launch_stream(StreamParams &p, const GemvJob &job, int K, int ntok, cudaStream_t st, int ctas = 0)
{
    static size_t attr_bytes[64];
    p.nmat = job.nmat;
    p.ntok = ntok;
    long long totalN = 0;
    for (int m = 0; m < job.nmat; ++m) {
        p.W[m] = static_cast<const uint8_t *>(job.W[m]);
        p.y[m] = job.y[m];
        p.N[m] = job.N[m];
        totalN += job.N[m];
    }
    const int sms = ctas > 0 ? ctas : num_sms();
    if (!plan_stream<FMT, NT>(p, K, totalN, sms)) return cudaErrorInvalidValue;
    p.gstart[0] = 0;
    for (int m = 0; m < kMaxMats; ++m)
        p.gstart[m + 1] = p.gstart[m] + (m < job.nmat ? (job.N[m] + p.R - 1) / p.R : 0);
    p.total_groups = p.gstart[job.nmat];
    p.status = device_status_word();
    const SmemLayout L(K, p.stage_alloc, NT, FMT == kFmtQ6K);
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (attr_bytes[dev] < L.total) {
        cudaError_t e = cudaFuncSetAttribute(kq_gemv_stream_kernel<FMT, NT>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.total);
        if (e != cudaSuccess) return e;
        attr_bytes[dev] = L.total;
    }
    const int grid = p.total_groups < sms ? p.total_groups : sms;
    return launch_pdl(kq_gemv_stream_kernel<FMT, NT>, dim3(grid), dim3(kThreads), L.total, st, p);
}

// Whether the NT-token staging of K activations leaves room for the stages.
template <int FMT, int NT>
bool staging_fits(int K)
{
    constexpr int kBytes = Fmt<FMT>::kBytes;
    constexpr uint32_t kSlack = (kBytes % 16) ? 32 : 0;
    return SmemLayout(K, 0, NT, FMT == kFmtQ6K).total + (size_t)kStages * align_up(kBytes + kSlack, 128) <=
           (size_t)kSmemLimit;
}

// B tokens of Q8_1 codes (planar [B][K]) against one matrix: one launch for
// B = 1, else launches of up to four tokens each (one token each when four
// tokens' staging does not fit in shared memory).
template <int FMT>
cudaError_t launch_tokens(const void *W, int N, int K, zq_q8_1 a, int B, float *y, cudaStream_t st)
{
    GemvJob job{};
    job.nmat = 1;
    job.W[0] = W;
    job.N[0] = N;
    const int per = (B > 1 && staging_fits<FMT, 4>(K)) ? 4 : 1;
    for (int t0 = 0; t0 < B; t0 += per) {
        const int nt = B - t0 < per ? B - t0 : per;
        StreamParams p{};
        p.qs = a.qs + (size_t)t0 * K;
        p.d = reinterpret_cast<const __half *>(a.d) + (size_t)t0 * (K / 32);
        p.s = reinterpret_cast<const __half *>(a.s) + (size_t)t0 * (K / 32);
        job.y[0] = y + (size_t)t0 * N;
        const cudaError_t e = (per == 1) ? launch_stream<FMT, 1>(p, job, K, 1, st)
                                         : launch_stream<FMT, 4>(p, job, K, nt, st);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// One token given as x and gamma: RMSNorm + Q8_1 inside the launch.
template <int FMT>
cudaError_t launch_fused(const GemvJob &job, int K, const float *x, const float *gamma, float eps, bool silu,
                         const zq_q8_1 *q8out, const void *pf, size_t pf_bytes, cudaStream_t st)
{
    StreamParams p{};
    p.x = x;
    p.gamma = gamma;
    p.eps = eps;
    p.silu = silu ? 1 : 0;
    if (q8out) p.q8out = *q8out;
    p.pf = static_cast<const uint8_t *>(pf);
    p.pf_bytes = pf_bytes;
    return launch_stream<FMT, 1>(p, job, K, 1, st);
}

}  // namespace stream
}  // namespace zq
