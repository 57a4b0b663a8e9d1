// q4k_gemm_tc.cu -- batched Q4_K x Q8_1 projections (placeholder dispatch to
// the dp4a kernels until the tensor-core kernels land).
#include "zq_internal.cuh"

namespace zq {

size_t gemm_tc_workspace_bytes(int N, int K, int B) { (void)N; (void)K; (void)B; return 0; }

cudaError_t launch_gemm_tc_wide(const void *W, int N, int K, zq_q8_1 a, int B, float *y,
                                int32_t *isums, void *ws, cudaStream_t st)
{
    (void)ws;
    if (isums) return cudaErrorNotSupported;
    return launch_gemv(W, nullptr, N, K, a, B, y, nullptr, nullptr, st);
}

cudaError_t launch_gemm_tc_narrow(const void *W, int N, int K, zq_q8_1 a, int B, float *y,
                                  int32_t *isums, void *ws, cudaStream_t st)
{
    (void)ws;
    if (isums) return cudaErrorNotSupported;
    return launch_gemv(W, nullptr, N, K, a, B, y, nullptr, nullptr, st);
}

}  // namespace zq
