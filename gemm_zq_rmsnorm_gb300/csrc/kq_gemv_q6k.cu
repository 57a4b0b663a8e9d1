// kq_gemv_q6k.cu -- the Q6_K instances of the streamed mat-vec
// (kq_gemv_stream.cuh): B = 1 .. 16 tokens of Q8_1 codes, or one token with
// RMSNorm + Q8_1 packing inside the launch.
//
// MIInfer README, "Status": MMVQ-style Q6_K x Q8_1 LM head; "Current phase":
// resident quantized Q6_K multi-token projection.
#include "kq_gemv_stream.cuh"

namespace zq {

cudaError_t launch_q6k_tokens(const void *W, int N, int K, zq_q8_1 a, int B, float *y, cudaStream_t st)
{
    return stream::launch_tokens<stream::kFmtQ6K>(W, N, K, a, B, y, st);
}

cudaError_t launch_q6k_fused(const GemvJob &job, int K, const float *x, const float *gamma, float eps,
                             const zq_q8_1 *q8out, cudaStream_t st)
{
    return stream::launch_fused<stream::kFmtQ6K>(job, K, x, gamma, eps, false, q8out, nullptr, 0, st);
}

}  // namespace zq
