/*
 * zq.h -- C ABI of the GB300 (sm_103a) quantized-projection library libzq.so.
 *
 * The library computes one hot path of LLM inference on one GPU:
 *   1. zq_rmsnorm_q8_1   RMSNorm of each token fused with Q8_1 packing of the
 *                        normalised activations;
 *   2. zq_q4k_gemv       Q4_K weight matrix x one Q8_1 token (decode, B = 1);
 *   3. zq_q4k_gemv_pair  two Q4_K matrices (FFN gate and up) x one token,
 *                        sharing one read of the activations;
 *   4. zq_q4k_gemm       Q4_K matrix x B Q8_1 tokens (chunked prefill B = 2..16,
 *                        full prefill e.g. B = 512) on the tensor cores.
 *
 * Sources: ZINC docs "ROCm backend", section "Build and verify" (RMS norm and
 * Q8 activation packing in one per-token kernel; hot Q4_K projections on
 * packed Q8 activations; paired Q4 gate/up projections; the engine's kernels
 * sit behind a C ABI); MIInfer README, "Status" (Q4_K x Q8_1 MMVQ-style
 * projections, Q4_K metadata staging, packed int8 dot4) and "Current phase"
 * (token-batched B = 4 chunk projections; int8 GEMM and tensor-core prefill).
 *
 * ---------------------------------------------------------------- formats
 * Q8_1 activations (planar, caller-owned device memory):
 *   qs : int8     [B][K]     codes q, |q| <= 127
 *   d  : binary16 [B][K/32]  per-32-block scale d = max|xh| / 127
 *   s  : binary16 [B][K/32]  per-32-block d * sum(q)
 *   q = round-half-away-from-zero(xh * (1/d)) computed in fp32 with the fp32 d;
 *   the stored d and s are that fp32 d and s rounded to binary16 (RNE).
 * Q4_K weights, N rows x K columns (K % 256 == 0), row-major, row n holding
 * K/256 consecutive 144-byte super-blocks of 256 weights:
 *   bytes 0..1 d, 2..3 dmin (binary16, little-endian);
 *   bytes 4..15 S[12]: eight 6-bit scales sc[j] and mins m[j]:
 *     j < 4 : sc = S[j] & 63,  m = S[j+4] & 63
 *     j >= 4: sc = (S[j+4] & 15) | (S[j-4] >> 6) << 4,
 *             m  = (S[j+4] >> 4) | (S[j]   >> 6) << 4
 *   bytes 16..143: weight i (0..31) of sub-block j at byte 32*(j/2)+i,
 *     low nibble for even j, high nibble for odd j;
 *   weight = d*sc[j]*q - dmin*m[j].
 * Output y (fp32, [B][N], token-major):
 *   y[t][n] = sum_{b,j} d_b*sc_j*d8_{t,bj}*I_{t,n,b,j} - dmin_b*m_j*s8_{t,bj},
 *   I = exact integer sum over the sub-block's 32 weights of q4*q8.
 *
 * ---------------------------------------------------------------- conventions
 * - All tensor pointers are caller-owned DEVICE memory.  The library never
 *   allocates device memory; it keeps no state except per-device launch
 *   configuration set up on the first call, and a thread-local error string.
 * - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *   stream).  Every call is asynchronous on that stream; none synchronises.
 * - Alignment: every tensor pointer must be 16-byte aligned.
 * - Outputs must not alias inputs.
 * - Every call returns ZQ_OK (0) or a negative status, checked on the host
 *   before anything is launched (argument, shape and alignment errors launch
 *   nothing).  zq_last_error() gives a one-line description of the last
 *   failure on the calling thread.
 * - Calls may be captured in a CUDA graph after one uncaptured call of the
 *   same entry point on the device (the first call sets kernel attributes).
 * - Kernels are launched with programmatic dependent launch: each may start
 *   while the previous kernel on the stream finishes, and waits for it before
 *   it reads activations or writes outputs.  Weights -- W, and gamma of the
 *   fused RMSNorm calls -- are read before that wait, so they must be complete
 *   in memory before the call is made (weights loaded at start-up are; a
 *   kernel that rewrites them needs a stream or event synchronisation first).
 */
#ifndef ZQ_H
#define ZQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ZQ_VERSION 1

#if defined(__GNUC__)
#define ZQ_API __attribute__((visibility("default")))
#else
#define ZQ_API
#endif

enum {
    ZQ_OK = 0,
    ZQ_ERR_ARG = -1,         /* null pointer, non-positive size, bad eps      */
    ZQ_ERR_SHAPE = -2,       /* K not a multiple of 256 (32 for the norm),    */
                             /* B or N out of range                           */
    ZQ_ERR_ALIGN = -3,       /* a tensor pointer not 16-byte aligned          */
    ZQ_ERR_CUDA = -4,        /* CUDA runtime error at launch                  */
    ZQ_ERR_DEVICE = -5,      /* device is not sm_103 / no device              */
    ZQ_ERR_WORKSPACE = -6    /* workspace missing or smaller than required    */
};

/* Planar Q8_1 activations of B tokens x K features (see "formats"). */
typedef struct zq_q8_1 {
    int8_t *qs;    /* [B][K]    */
    uint16_t *d;   /* [B][K/32] binary16 bits */
    uint16_t *s;   /* [B][K/32] binary16 bits */
} zq_q8_1;

/*
 * Fused RMSNorm + Q8_1 packing (ZINC docs "ROCm backend", "Build and verify":
 * normalisation and Q8 packing share one per-token kernel).
 *   x     : fp32 [B][K] input activations
 *   gamma : fp32 [K]    RMSNorm weight
 *   eps   : >= 0, added to the mean square
 *   out   : Q8_1 [B][K] (qs, d, s written)
 * xh_k = (x_k * r) * gamma_k, r = 1 / sqrt(ss/K + eps); each step one IEEE
 * fp32 operation, ss summed in this fixed order: per 32-block a fused
 * multiply-add chain over its squares in index order; 256 slots, slot t
 * summing the block partials b = t (mod 256) in increasing b; then the
 * pairwise tree slot[t] += slot[t+off] for off = 128, 64, ..., 1.
 * Shapes: B >= 1, K >= 32, K % 32 == 0, K <= 1048576.
 */
ZQ_API int zq_rmsnorm_q8_1(const float *x, const float *gamma, int B, int K, float eps,
                    zq_q8_1 out, void *stream);

/*
 * Decode mat-vec, one token (MIInfer README, "Status": Q4_K x Q8_1 MMVQ-style
 * projection; ZINC docs "ROCm backend": packed Q8 activations for Q4_K).
 *   W : Q4_K [N][K/256] super-blocks (N*K/256*144 bytes)
 *   a : Q8_1 of one token (K features)
 *   y : fp32 [N]
 * Shapes: N >= 1, K >= 256, K % 256 == 0.
 */
ZQ_API int zq_q4k_gemv(const void *W, int N, int K, zq_q8_1 a, float *y, void *stream);

/*
 * Paired decode mat-vec for FFN gate and up (ZINC docs "ROCm backend":
 * paired Q4 projections; MIInfer README, "Status": shared Q4_K x Q8_1 FFN
 * gate/up path).  Both matrices are N x K Q4_K; one activation read serves
 * both.  y_gate = Wg a, y_up = Wu a (fp32 [N] each).
 */
ZQ_API int zq_q4k_gemv_pair(const void *Wg, const void *Wu, int N, int K, zq_q8_1 a,
                     float *y_gate, float *y_up, void *stream);

/*
 * Decode mat-vec of up to four matrices that read the same Q8_1 input, in one
 * launch (ZINC docs "ROCm backend": Q8 activations packed once and reused by
 * the Q4_K projections that follow; MIInfer README, "Status": shared
 * activation staging).  The q/k/v projections of a layer are the intended use.
 *   nmat : 1..4;  W[m] : Q4_K N[m] x K (16-byte aligned);  y[m] : fp32 [N[m]]
 *   (16-byte aligned);  W, N, y are host arrays of nmat entries.
 * Each y[m] equals zq_q4k_gemv(W[m], N[m], K, a, y[m]) bit for bit.  Shapes as
 * zq_q4k_gemv; K > 32768 runs one launch per matrix.
 */
ZQ_API int zq_q4k_gemv_multi(int nmat, const void *const *W, const int *N, int K, zq_q8_1 a,
                             float *const *y, void *stream);

/*
 * Fused decode step: RMSNorm and Q8_1 packing of one token x (as
 * zq_rmsnorm_q8_1 with B = 1), then y[m] = W[m] (Q8_1 of x) for up to four
 * matrices, in one launch (ZINC docs "ROCm backend", "Build and verify":
 * normalisation and Q8 packing fused ahead of the Q4 projections).  Every
 * thread block computes the codes itself in shared memory in the canonical
 * order, so they are byte for byte those of zq_rmsnorm_q8_1 and each y[m]
 * equals zq_q4k_gemv on them bit for bit.  The normalised input never goes
 * through device memory unless q8_out (optional, may be NULL; planes of one
 * token) asks for it.
 *   x, gamma : fp32 [K], 16-byte aligned;  eps >= 0;
 *   nmat, W, N, y : as zq_q4k_gemv_multi;
 *   l2_prefetch, l2_prefetch_bytes : optional (NULL / 0): device bytes the
 *     caller's next launch will read (the next projection's weights); once
 *     its own weights are requested, the kernel pulls them into L2 so that the
 *     next launch starts on L2 hits.  16-byte aligned; a hint, never read by
 *     this call's arithmetic.
 * Shapes: K % 256 == 0, 256 <= K <= 32768 (larger K: ZQ_ERR_SHAPE).
 */
ZQ_API int zq_rmsnorm_q4k_gemv(const float *x, const float *gamma, float eps, int K, int nmat,
                               const void *const *W, const int *N, float *const *y,
                               const zq_q8_1 *q8_out, const void *l2_prefetch,
                               size_t l2_prefetch_bytes, void *stream);

/*
 * Batched projection of B tokens (MIInfer README, "Current phase":
 * token-batched chunk projections and tensor-core/int8 GEMM prefill).
 *   W : Q4_K N x K;  a : Q8_1 of B tokens;  y : fp32 [B][N].
 *   workspace / workspace_bytes : caller-owned device scratch of at least
 *     zq_q4k_gemm_workspace_bytes(N, K, B) bytes (may be NULL when that is 0,
 *     as it is for B = 1 and for 2 <= B <= 4 with K <= 32768; at least
 *     4*B*K + 4*B + B*K/8, each part rounded up to 256, otherwise).  It holds
 *     the activations the tensor cores read (each Q8_1 value q8*d8 split into
 *     two binary16 numbers), a per-token scale, the scaled block sums and
 *     partial sums; its contents on entry do not matter and are not
 *     preserved.
 * B = 1 runs the decode mat-vec; 2 <= B <= 4 (K <= 32768) the same streamed
 * kernel with the tokens staged together, each decoded weight used for all of
 * them (the workspace is not touched).  5 <= B <= 16 runs the chunk kernel
 * (CTA pairs: 256 weight rows x the 16 tokens' hi and lo parts per MMA),
 * B >= 17 the prefill kernel (CTA pairs: 256 weight rows x 256 tokens).
 * There every product of an activation part and a weight code sc*q4 is exact
 * and the products are summed in fp32 per 256-weight super-block, then
 * scaled by d_b (the min term, by dmin_b, enters the same sum) in fp32.
 * Shapes: 1 <= B <= 65536, N >= 1, K % 256 == 0, K >= 256.
 */
ZQ_API int zq_q4k_gemm(const void *W, int N, int K, zq_q8_1 a, int B, float *y,
                void *workspace, size_t workspace_bytes, void *stream);

/*
 * zq_q4k_gemm for callers that cannot provide device memory.  (No counterpart
 * on the pages this library follows: it is an interface for integration.)
 * Some callers have no device memory to pass when they call: engines that
 * carve every byte of device memory out of one arena at start-up and allow
 * no allocation afterwards, and plugins run by a host framework that offers
 * them no allocator.  This entry point computes what zq_q4k_gemm computes
 * (the same kernels, one K range per output tile) but takes its scratch from
 * a fixed device array inside the library instead of a workspace argument,
 * and never calls cudaMalloc, cudaFree or any allocating routine.
 *   - Limit: the scratch (4*B*K + B*K/8 + 4*B bytes, each part padded to
 *     256 bytes) must fit in the array (42 MiB + 256 KiB), i.e.
 *     B*K <= 10485760 (for example B = 512 with K up to 20480); larger
 *     shapes return ZQ_ERR_WORKSPACE without launching.  B = 1 needs no
 *     scratch.
 *   - Every GPU that loads the library holds the 42 MiB array until the
 *     process exits.
 *   - The first call on a device looks up the array's device address (once per
 *     device, with that device current); make that first call before any
 *     stream capture.
 *   - All calls share the one array and it keeps the previous call's contents
 *     (each call overwrites what it reads).  Calls whose kernels overlap on the
 *     GPU -- on different streams, or from several host threads without
 *     ordering -- race on it: order them on one stream.
 */
ZQ_API int zq_q4k_gemm_noalloc(const void *W, int N, int K, zq_q8_1 a, int B, float *y,
                               void *stream);

/*
 * SiLU(gate) * up packed to Q8_1: the input of the FFN down projection
 * (MIInfer README, "Current phase": a fused SiLU(gate)*up epilogue feeding the
 * down projection).  h = silu(gate) * up with silu(g) = g / (1 + exp(-g)); the
 * pages fix no precision, so every step is one IEEE fp32 operation of this
 * library's definition -- exp(a) for a clamped to [-86, 88] as rint-based
 * range reduction with ln 2 in two parts, a degree-7 Taylor polynomial of
 * e^r in fma Horner form with coefficients 1/n! rounded to fp32, and an exact
 * power-of-two scaling -- and h is packed exactly as zq_rmsnorm_q8_1 packs xh.
 *   gate, up : fp32 [B][K] (16-byte aligned);  out : Q8_1 planes of B x K.
 * Shapes: B >= 1, K % 32 == 0.
 */
ZQ_API int zq_silu_mul_q8_1(const float *gate, const float *up, int B, int K, zq_q8_1 out,
                            void *stream);

/*
 * Fused down-projection step: the Q8_1 of silu(gate) * up (as
 * zq_silu_mul_q8_1 with B = 1, byte for byte) computed inside the mat-vec
 * kernel, then y[m] = W[m] h for up to four matrices, in one launch.
 *   gate, up : fp32 [K];  nmat, W, N, y, q8_out, l2_prefetch : as
 *   zq_rmsnorm_q4k_gemv.  Shapes: K % 256 == 0, 256 <= K <= 32768.
 */
ZQ_API int zq_silu_q4k_gemv(const float *gate, const float *up, int K, int nmat,
                            const void *const *W, const int *N, float *const *y,
                            const zq_q8_1 *q8_out, const void *l2_prefetch,
                            size_t l2_prefetch_bytes, void *stream);

/*
 * Q4_K weights dequantised to binary16, for a dequantise-then-GEMM prefill
 * (MIInfer README, "Current phase": 16-bit dequantised weights ahead of a
 * dense GEMM).  The library's own projections do not use it; it lets that
 * design be measured beside them.
 *   W : Q4_K N x K;  out : binary16 [N][K] (device, 16-byte aligned, 2*N*K bytes).
 * Per weight, in fp32: a = d*sc, b = dmin*m (exact), w = a*q - b (one
 * rounding), then w rounded to binary16 (nearest even).
 */
ZQ_API int zq_q4k_dequant_f16(const void *W, int N, int K, void *out, void *stream);

/*
 * Q8_1 activations dequantised to binary16, the activation half of the
 * dequantise-then-GEMM design (MIInfer README, "Current phase").
 *   a : Q8_1 planes of B tokens x K;  out : binary16 [B][K] (device, 16-byte
 *   aligned, 2*B*K bytes).  x = q8 * d8 in fp32 (exact), rounded to binary16
 *   (nearest even).  K % 32 == 0.
 */
ZQ_API int zq_q8_1_dequant_f16(zq_q8_1 a, int B, int K, void *out, void *stream);

/*
 * Dense binary16 GEMM on the tensor cores, the GEMM half of the
 * dequantise-then-GEMM design (MIInfer README, "Current phase": Q4_K
 * dequantised to 16-bit weights ahead of a dense GEMM), measured beside the
 * library's Q4_K x Q8_1 projection; no library GEMM is involved.
 *   W16 : binary16 [N][K] (row-major, device);  X16 : binary16 [B][K];
 *   y   : fp32 [B][N] (device), y[t][n] = sum_k X16[t][k] * W16[n][k], each
 *         product exact, accumulated in fp32 (order unspecified);
 *   workspace : device, at least zq_f16_gemm_workspace_bytes(N, K, B) bytes
 *         (split-K partial sums; 0 bytes when the call does not split).
 * All pointers 16-byte aligned; K % 64 == 0, 1 <= B <= 65536.
 */
ZQ_API size_t zq_f16_gemm_workspace_bytes(int N, int K, int B);
ZQ_API int zq_f16_gemm(const void *W16, int N, int K, const void *X16, int B, float *y, void *workspace,
                       size_t workspace_bytes, void *stream);

/*
 * ---------------------------------------------------------- Q5_K and Q6_K
 * The other k-quant blocks of a Q4_K_M checkpoint (MIInfer README, "Status":
 * Q5_K x Q8_1 MMVQ-style recurrent output projection, MMVQ-style Q6_K x Q8_1
 * LM head; "Current phase": Q5_K B = 4 reuse in layer-major prefill; ZINC
 * docs "ROCm backend": packed Q8 activations feed the hot Q4_K, Q5_K and Q6_K
 * projections).  N rows x K columns (K % 256 == 0), rows of K/256
 * consecutive super-blocks of 256 weights, rows consecutive:
 *   Q5_K, 176 bytes: bytes 0..15 as Q4_K (d, dmin, scales and mins);
 *     bytes 16..47 qh, bit j of byte 16+i = bit 4 of weight i of sub-block j;
 *     bytes 48..175 the low four bits, placed as the Q4_K nibbles;
 *     weight = d*sc[j]*q - dmin*m[j], q in 0..31.
 *   Q6_K, 210 bytes, sixteen sub-blocks of 16 weights; weight k has
 *     h = k/128, c = (k%128)/32, i = k%32:
 *     bytes 0..127 low four bits at byte 64h + 32(c%2) + i (low nibble for
 *     c < 2, high for c >= 2); bytes 128..191 top two bits at bits 2c, 2c+1
 *     of byte 128 + 32h + i; bytes 192..207 int8 scales sc[k/16];
 *     bytes 208..209 d (binary16);  weight = d*sc[k/16]*(q - 32), q in 0..63.
 *     Rows are 210*K/256 bytes: only the matrix start needs 16-byte alignment.
 * Output as for Q4_K: Q5_K y = sum_{b,j} d*sc_j*d8*I_j - dmin*m_j*s8 with
 * I_j over the 32 weights of sub-block j; Q6_K y = sum_{b,s} d*sc_s*d8*I_s
 * with I_s = sum of (q - 32)*q8 over the 16 weights of sub-block s (d8 of the
 * Q8_1 block holding them; s8 is not used).
 *
 * zq_q5k_gemm / zq_q6k_gemm: y [B][N] = W x B tokens of Q8_1 codes,
 *   1 <= B <= 16 (launches of up to four tokens; every weight read once per
 *   launch), 256 <= K <= 32768.  zq_q5k_gemv / zq_q6k_gemv: the same, B = 1.
 * zq_rmsnorm_q6k_gemv: one token given as x, gamma, eps (RMSNorm + Q8_1
 *   packing in the launch, byte for byte as zq_rmsnorm_q8_1), y [N] = W xh;
 *   the LM head after the final norm.  q8_out as for zq_rmsnorm_q4k_gemv.
 * Errors: as for the Q4_K calls; ZQ_ERR_SHAPE also for B outside [1, 16] or
 * K > 32768.  No workspace.
 */
ZQ_API int zq_q5k_gemm(const void *W, int N, int K, zq_q8_1 a, int B, float *y, void *stream);
ZQ_API int zq_q6k_gemm(const void *W, int N, int K, zq_q8_1 a, int B, float *y, void *stream);
ZQ_API int zq_q5k_gemv(const void *W, int N, int K, zq_q8_1 a, float *y, void *stream);
ZQ_API int zq_q6k_gemv(const void *W, int N, int K, zq_q8_1 a, float *y, void *stream);
ZQ_API int zq_rmsnorm_q6k_gemv(const float *x, const float *gamma, float eps, int K,
                               const void *W, int N, float *y, const zq_q8_1 *q8_out,
                               void *stream);
/* Storage sizes of N x K Q5_K and Q6_K matrices. */
ZQ_API size_t zq_q5k_bytes(int N, int K);
ZQ_API size_t zq_q6k_bytes(int N, int K);

/* Bytes of device workspace zq_q4k_gemm needs for this shape (0 if none). */
ZQ_API size_t zq_q4k_gemm_workspace_bytes(int N, int K, int B);

/*
 * RMSNorm + Q8_1 of B tokens and the batched projection in one call (ZINC
 * docs "ROCm backend", "Build and verify": RMS normalisation and Q8
 * activation packing in one per-token kernel; MIInfer README, "Current
 * phase": batched Q4_K projections).  y equals zq_rmsnorm_q8_1 followed by
 * zq_q4k_gemm on the same workspace, bit for bit; for B >= 5 the
 * normalisation kernel also writes the binary16 activation parts the tensor
 * cores read, saving a launch and a pass over the codes.
 *   x : fp32 [B][K];  gamma : fp32 [K];  eps >= 0;  W, N, y : as zq_q4k_gemm.
 *   q8_out : optional Q8_1 destination of the codes (required for
 *     2 <= B <= 4, where the streamed mat-vec reads them).
 *   workspace : zq_q4k_gemm_workspace_bytes(N, K, B) bytes.
 * Shapes: K % 256 == 0, 256 <= K <= 32768, 1 <= B <= 65536.
 */
ZQ_API int zq_rmsnorm_q4k_gemm(const float *x, const float *gamma, float eps, int B, int K, const void *W, int N,
                               float *y, const zq_q8_1 *q8_out, void *workspace, size_t workspace_bytes,
                               void *stream);

/* Storage sizes: N x K Q4_K matrix; Q8_1 planes of B x K (qs + d + s). */
ZQ_API size_t zq_q4k_bytes(int N, int K);
ZQ_API size_t zq_q8_1_bytes(int B, int K);

/*
 * Device-side error word of the current device, copied to *flags (host
 * memory; synchronous).  Bit 0 (ZQ_DEVICE_WAIT_EXPIRED): a bounded wait inside
 * a pipelined kernel gave up -- that kernel's outputs are invalid.  The
 * pipelined kernels never spin without a limit.  clear != 0 resets the word.
 */
#define ZQ_DEVICE_WAIT_EXPIRED 1u
ZQ_API int zq_device_status(unsigned int *flags, int clear);

/* Status text, last error on this thread, library version (ZQ_VERSION). */
ZQ_API const char *zq_status_string(int status);
ZQ_API const char *zq_last_error(void);
ZQ_API int zq_version(void);

/*
 * Test hook: exact sub-block integer sums I[t][n][K/32] (int32, device
 * memory) computed by the kernels' own inner products.  path = 0: the packed
 * dot4 (dp4a) inner product of the mat-vec kernels, any B; paths 1 (B >= 17)
 * and 2 (2 <= B <= 16): tcgen05 MMAs on the projection's tile layout, fp16
 * operands holding q8 and q4 exactly, one K = 32 accumulator per sub-block
 * read back from tensor memory.  Paths 1 and 2 need a device workspace of
 * at least 2*B*K bytes (the binary16 copy of the codes); path 0 none.
 */
ZQ_API int zq_debug_q4k_isums(const void *W, int N, int K, zq_q8_1 a, int B,
                       int32_t *isums, int path, void *workspace,
                       size_t workspace_bytes, void *stream);

/*
 * Test hook: the launch plan of the streamed mat-vec kernel (host-side, no
 * device needed) for weight format wtype (4, 5, 6 = Q4_K, Q5_K, Q6_K), ntok
 * tokens per launch (1 or 4), K columns, total_rows rows over all matrices of
 * the launch and sms CTAs.  out[8] (host memory) receives: rows per stage,
 * pieces per row, blocks per piece, segments per row, warp-local rows (0/1),
 * bytes per stage, dynamic shared memory per CTA, bytes per row.
 * ZQ_ERR_SHAPE when the staging does not fit (the calls then use one token
 * per launch) or the sizes are out of range.
 */
ZQ_API int zq_debug_stream_plan(int wtype, int ntok, int K, long long total_rows, int sms, int32_t *out);

/*
 * Throughput probe of the arithmetic the projection kernels can use on this
 * GPU (no counterpart on the pages; the rates are the denominators of the
 * prefill metric, because the int8 tcgen05 MMA, kind::i8, does not exist on
 * sm_103a).  One launch of `blocks` blocks, each thread or issuing thread
 * running `iters` steps; the caller times it.  Operations per launch:
 *   kind 0  dp4a (packed int8 dot products, 256 threads, 8 per step):
 *           blocks * 256 * iters * 8 * 8;
 *   kind 1  mma.sync m16n8k32 s8 (8 warps, 4 per step):
 *           blocks * 8 * iters * 4 * 2 * 16 * 8 * 32;
 *   kind 2  tcgen05.mma kind::f16 128 x 256 x 16 (one issuing thread per
 *           block, one block per SM at most): blocks * iters * 2*128*256*16;
 *   kinds 3, 4  the same MMA with N = 32 and N = 16 (the chunk shapes):
 *           blocks * iters * 2*128*N*16;
 *   kind 5  N = 32 with the A operand read from tensor memory:
 *           blocks * iters * 2*128*32*16;
 *   kind 6  N = 32, two warps of each block issuing at once (own
 *           accumulators): blocks * 2 * iters * 2*128*32*16;
 *   kind 7  CTA pairs (blocks rounded down to even), one thread per pair
 *           issuing 256 x 32 x 16 MMAs (cta_group::2):
 *           (blocks/2) * iters * 2*256*32*16;
 *   kinds 8, 9  as 3 and 7, with the issuing loop run by a whole warp and
 *           each MMA issued by one elected lane;
 *   kind 10 as 9 with the A operand read from tensor memory.
 *   sink : device memory of at least blocks * 256 ints (results kept live).
 * A kind-2 probe whose bounded wait expires sets ZQ_DEVICE_WAIT_EXPIRED.
 */
ZQ_API int zq_debug_peak_probe(int kind, int blocks, int iters, void *sink, void *stream);

/*
 * Test hook for the failure path of the bounded waits (no counterpart on the
 * pages): one launch of the streamed Q4_K mat-vec (one token of Q8_1 codes a,
 * N rows of K columns, y as in zq_q4k_gemv) on `ctas` CTAs (1 .. SM count)
 * whose copy producers stop before issuing their stage `withhold_stage`
 * (counted from 0 in each CTA), and whose waits give up after wait_us
 * microseconds (1 .. 2000000) instead of two seconds.  Every CTA with more
 * than withhold_stage stages of work then finds its consumers' wait expire,
 * raises ZQ_DEVICE_WAIT_EXPIRED in the device status word and returns; no copy
 * is in flight when it does.  Rows of the withheld and later stages of y are
 * left unwritten.  The call itself returns ZQ_OK (the expiry is reported by
 * zq_device_status, which the caller should then clear).  K <= 32768.
 */
ZQ_API int zq_debug_wait_expiry(const void *W, int N, int K, zq_q8_1 a, float *y, int withhold_stage,
                                unsigned int wait_us, int ctas, void *stream);

/*
 * Copy `bytes` bytes from src to dst with the GPU's SMs, on `stream`, ordered
 * after the stream's previous kernel (no counterpart on the pages: the host <->
 * device plumbing of a decode step, whose activations are a few hundred KB a
 * step and for which a copy engine's start-up latency dominates).  Each
 * pointer may be device memory of the current device, or pinned host memory
 * that the driver maps into the device's address space (cudaHostAlloc,
 * cudaHostRegister; on a Grace-coupled GPU the SMs reach it over the
 * chip-to-chip link).  Both are checked with cudaPointerGetAttributes before
 * anything runs: any other pointer (pageable host memory, another device's
 * memory, an unknown address) returns ZQ_ERR_ARG.  The caller owns both
 * buffers, which must hold `bytes` bytes and must not overlap; any alignment
 * works (16-byte aligned pointers copy 16 bytes per access).  bytes = 0 does
 * nothing and returns ZQ_OK.
 */
ZQ_API int zq_copy(void *dst, const void *src, size_t bytes, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* ZQ_H */
