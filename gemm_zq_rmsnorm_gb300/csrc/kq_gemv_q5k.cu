// kq_gemv_q5k.cu -- the Q5_K instances of the streamed mat-vec
// (kq_gemv_stream.cuh): B = 1 .. 16 tokens of Q8_1 codes.
//
// MIInfer README, "Status": Q5_K x Q8_1 MMVQ-style recurrent output projection
// (scale/min hoisting, paired nibbles); "Current phase": shape-specific Q5_K
// B=4 reuse in layer-major prefill.
#include "kq_gemv_stream.cuh"

namespace zq {

cudaError_t launch_q5k_tokens(const void *W, int N, int K, zq_q8_1 a, int B, float *y, cudaStream_t st)
{
    return stream::launch_tokens<stream::kFmtQ5K>(W, N, K, a, B, y, st);
}

}  // namespace zq
