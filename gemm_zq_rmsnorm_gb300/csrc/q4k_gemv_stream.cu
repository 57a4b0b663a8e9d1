// q4k_gemv_stream.cu -- the Q4_K instance of the streamed decode mat-vec
// (kq_gemv_stream.cuh): plain, paired and up-to-four-matrix launches, with
// Q8_1 input or with RMSNorm (or SiLU(gate)*up) + Q8_1 packing in the launch;
// and small batches of tokens (launches of four) for the chunked prefill.
//
// MIInfer README, "Status": Q4_K x Q8_1 MMVQ-style projections (FFN down,
// shared gate/up; Q4_K metadata staging; packed int8 dot4).  ZINC docs "ROCm
// backend", "Build and verify": paired Q4 projections; RMS normalization and
// Q8 activation packing in one per-token kernel.
#include "kq_gemv_stream.cuh"

namespace zq {

bool gemv_stream_supported(int K) { return K <= stream::kMaxK; }

cudaError_t launch_gemv_stream(const GemvJob &job, int K, zq_q8_1 a, cudaStream_t st)
{
    stream::StreamParams p{};
    p.qs = a.qs;
    p.d = reinterpret_cast<const __half *>(a.d);
    p.s = reinterpret_cast<const __half *>(a.s);
    return stream::launch_stream<stream::kFmtQ4K, 1>(p, job, K, 1, st);
}

cudaError_t launch_q4k_tokens(const void *W, int N, int K, zq_q8_1 a, int B, float *y, cudaStream_t st)
{
    return stream::launch_tokens<stream::kFmtQ4K>(W, N, K, a, B, y, st);
}

cudaError_t launch_gemv_stream_fused(const GemvJob &job, int K, const float *x, const float *gamma, float eps,
                                     bool silu, const zq_q8_1 *q8out, const void *pf, size_t pf_bytes,
                                     cudaStream_t st)
{
    return stream::launch_fused<stream::kFmtQ4K>(job, K, x, gamma, eps, silu, q8out, pf, pf_bytes, st);
}

// Failure-path test: one matrix, one token, on `ctas` CTAs, whose producers
// withhold stage `withhold` (counted per CTA from 0) and whose waits give up
// after wait_ns.
cudaError_t launch_q4k_wait_expiry(const void *W, int N, int K, zq_q8_1 a, float *y, int withhold,
                                   uint64_t wait_ns, int ctas, cudaStream_t st)
{
    GemvJob job{};
    job.nmat = 1;
    job.W[0] = W;
    job.N[0] = N;
    job.y[0] = y;
    stream::StreamParams p{};
    p.qs = a.qs;
    p.d = reinterpret_cast<const __half *>(a.d);
    p.s = reinterpret_cast<const __half *>(a.s);
    p.wait_ns = wait_ns;
    p.withhold = withhold + 1;
    return stream::launch_stream<stream::kFmtQ4K, 1>(p, job, K, 1, st, ctas);
}

// Launch plan of the streamed kernel (host only): out = R, P, CB, nseg,
// warp-local, stage bytes, dynamic shared memory, row bytes.
bool stream_plan_query(int fmt, int nt, int K, long long total_rows, int sms, int32_t *out)
{
    stream::StreamParams p{};
    bool ok = false;
    size_t smem = 0;
    auto run = [&](auto plan, auto smem_of) {
        ok = plan(p, K, total_rows, sms);
        if (ok) smem = smem_of(p);
    };
    if (fmt == 4 && nt == 1) run(stream::plan_stream<stream::kFmtQ4K, 1>, stream::plan_smem<stream::kFmtQ4K, 1>);
    else if (fmt == 4 && nt == 4) run(stream::plan_stream<stream::kFmtQ4K, 4>, stream::plan_smem<stream::kFmtQ4K, 4>);
    else if (fmt == 5 && nt == 1) run(stream::plan_stream<stream::kFmtQ5K, 1>, stream::plan_smem<stream::kFmtQ5K, 1>);
    else if (fmt == 5 && nt == 4) run(stream::plan_stream<stream::kFmtQ5K, 4>, stream::plan_smem<stream::kFmtQ5K, 4>);
    else if (fmt == 6 && nt == 1) run(stream::plan_stream<stream::kFmtQ6K, 1>, stream::plan_smem<stream::kFmtQ6K, 1>);
    else if (fmt == 6 && nt == 4) run(stream::plan_stream<stream::kFmtQ6K, 4>, stream::plan_smem<stream::kFmtQ6K, 4>);
    else return false;
    if (!ok) return false;
    const int32_t v[8] = {p.R, p.P, p.CB, p.nseg, p.wl, (int32_t)p.stage_alloc, (int32_t)smem, (int32_t)p.rowbytes};
    for (int i = 0; i < 8; ++i) out[i] = v[i];
    return true;
}

}  // namespace zq
