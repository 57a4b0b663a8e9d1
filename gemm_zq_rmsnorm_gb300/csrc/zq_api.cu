// zq_api.cu -- the C ABI of libzq.so: argument, shape and alignment checks,
// device checks, dispatch by batch size, status codes and error text.
//
// ZINC docs "ROCm backend", "Build and verify": the engine keeps its GPU
// kernels behind a C ABI; every fused path is selectable, and a request the
// build cannot serve fails instead of falling back (Zynfer README: forced
// unsupported paths exit with an error).  Nothing here computes: every step of
// the path runs in the kernels of the other translation units.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "zq_internal.cuh"
#include "zq_tc_common.cuh"

__device__ unsigned int g_zq_device_status;

namespace zq {

namespace {
thread_local std::string g_last_error;

constexpr int kMaxDevices = 64;
int g_sms[kMaxDevices];
bool g_checked[kMaxDevices];
int g_dev_status[kMaxDevices];
unsigned int *g_status_word[kMaxDevices];
std::mutex g_mu;

int fail(int status, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
int fail(int status, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return status;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device check, once per device: the kernels are built for sm_103a only.
int check_device(int *dev_out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(ZQ_ERR_DEVICE, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(ZQ_ERR_DEVICE, "device index %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_checked[dev]) {
        int major = 0, minor = 0, sms = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        g_sms[dev] = sms;
        g_dev_status[dev] = (major == 10 && minor == 3) ? ZQ_OK : ZQ_ERR_DEVICE;
        if (g_dev_status[dev] == ZQ_OK) {
            void *w = nullptr;
            if (cudaGetSymbolAddress(&w, g_zq_device_status) != cudaSuccess) {
                cudaGetLastError();
                return fail(ZQ_ERR_DEVICE, "device %d: cannot resolve the device status word", dev);
            }
            g_status_word[dev] = static_cast<unsigned int *>(w);
        }
        g_checked[dev] = true;
    }
    *dev_out = dev;
    if (g_dev_status[dev] != ZQ_OK)
        return fail(ZQ_ERR_DEVICE, "device %d is not sm_103 (GB300); libzq is built for sm_103a only", dev);
    return ZQ_OK;
}

// The device address of p when the device may access it: memory of this
// device (or managed memory), or pinned host memory mapped into the device's
// address space; anything else is refused before a kernel could touch it.
int device_address(const void *p, int dev, void **out, const char *what)
{
    cudaPointerAttributes a;
    const cudaError_t e = cudaPointerGetAttributes(&a, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(ZQ_ERR_ARG, "%s: pointer unknown to CUDA (%s)", what, cudaGetErrorString(e));
    }
    if ((a.type == cudaMemoryTypeDevice && a.device == dev) || a.type == cudaMemoryTypeManaged) {
        *out = a.devicePointer ? a.devicePointer : const_cast<void *>(p);
        return ZQ_OK;
    }
    if (a.type == cudaMemoryTypeHost && a.devicePointer != nullptr) {
        *out = a.devicePointer;
        return ZQ_OK;
    }
    return fail(ZQ_ERR_ARG, "%s: neither memory of device %d nor pinned host memory mapped into it", what, dev);
}

int launched(cudaError_t e, const char *what)
{
    if (e != cudaSuccess) return fail(ZQ_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    return ZQ_OK;
}

int check_q8(const zq_q8_1 &a, const char *name)
{
    if (!a.qs || !a.d || !a.s) return fail(ZQ_ERR_ARG, "%s: null Q8_1 plane", name);
    if (!aligned16(a.qs) || !aligned16(a.d) || !aligned16(a.s))
        return fail(ZQ_ERR_ALIGN, "%s: Q8_1 planes must be 16-byte aligned", name);
    return ZQ_OK;
}

// Batches of up to four tokens run on the streamed mat-vec (every weight read
// once, four tokens per decoded weight): measured 1.6-2.5x faster than the
// tensor-core small-batch kernel at B = 2..4 on the chunk shapes, slower from
// B = 8 (two launches).
bool chunk_streams(int B, int K) { return B >= 2 && B <= 4 && gemv_stream_supported(K); }

int check_q4k(const void *W, int N, int K, const char *name)
{
    if (!W) return fail(ZQ_ERR_ARG, "%s: null weight pointer", name);
    if (!aligned16(W)) return fail(ZQ_ERR_ALIGN, "%s: weights must be 16-byte aligned", name);
    if (N < 1) return fail(ZQ_ERR_SHAPE, "%s: N = %d must be >= 1", name, N);
    if (K < 256 || K % 256 != 0 || K > (1 << 22))
        return fail(ZQ_ERR_SHAPE, "%s: K = %d must be a positive multiple of 256 (<= 2^22)", name, K);
    return ZQ_OK;
}

}  // namespace

unsigned int *device_status_word()
{
    int dev = 0;
    cudaGetDevice(&dev);
    return (dev >= 0 && dev < kMaxDevices) ? g_status_word[dev] : nullptr;
}

cudaError_t launch_gemv_dispatch(const void *W, const void *W2, int N, int K, zq_q8_1 a, float *y,
                                 float *y2, cudaStream_t st)
{
    if (gemv_stream_supported(K)) {
        GemvJob job{};
        job.nmat = W2 ? 2 : 1;
        job.W[0] = W;
        job.N[0] = N;
        job.y[0] = y;
        if (W2) {
            job.W[1] = W2;
            job.N[1] = N;
            job.y[1] = y2;
        }
        return launch_gemv_stream(job, K, a, st);
    }
    return launch_gemv(W, W2, N, K, a, 1, y, y2, nullptr, st);
}

// SM count of the current device, read once per device; launch shapes and
// workspace sizes derive from it, so the workspace query and the call agree.
int num_sms()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return 148;
    }
    if (g_sms[dev] <= 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) {
            cudaGetLastError();
            return 148;
        }
        g_sms[dev] = v;
    }
    return g_sms[dev];
}

}  // namespace zq

using namespace zq;

extern "C" {

int zq_version(void) { return ZQ_VERSION; }

const char *zq_last_error(void) { return g_last_error.c_str(); }

const char *zq_status_string(int status)
{
    switch (status) {
    case ZQ_OK: return "ok";
    case ZQ_ERR_ARG: return "invalid argument";
    case ZQ_ERR_SHAPE: return "unsupported shape";
    case ZQ_ERR_ALIGN: return "misaligned pointer";
    case ZQ_ERR_CUDA: return "CUDA error";
    case ZQ_ERR_DEVICE: return "unsupported or missing device";
    case ZQ_ERR_WORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
    }
}

size_t zq_q4k_bytes(int N, int K)
{
    if (N < 1 || K < 256 || K % 256) return 0;
    return (size_t)N * (size_t)(K / 256) * kQ4KBlockBytes;
}

size_t zq_q8_1_bytes(int B, int K)
{
    if (B < 1 || K < 32 || K % 32) return 0;
    return (size_t)B * K + 2 * sizeof(uint16_t) * (size_t)B * (K / 32);
}

int zq_rmsnorm_q8_1(const float *x, const float *gamma, int B, int K, float eps, zq_q8_1 out,
                    void *stream)
{
    if (!x || !gamma) return fail(ZQ_ERR_ARG, "zq_rmsnorm_q8_1: null x or gamma");
    if (!aligned16(x) || !aligned16(gamma))
        return fail(ZQ_ERR_ALIGN, "zq_rmsnorm_q8_1: x and gamma must be 16-byte aligned");
    if (!(eps >= 0.0f) || eps != eps) return fail(ZQ_ERR_ARG, "zq_rmsnorm_q8_1: eps must be >= 0");
    if (B < 1 || B > (1 << 24)) return fail(ZQ_ERR_SHAPE, "zq_rmsnorm_q8_1: B = %d out of range", B);
    if (K < 32 || K % 32 != 0 || K > (1 << 20))
        return fail(ZQ_ERR_SHAPE, "zq_rmsnorm_q8_1: K = %d must be a multiple of 32 in [32, 2^20]", K);
    int st = check_q8(out, "zq_rmsnorm_q8_1");
    if (st) return st;
    int dev;
    if ((st = check_device(&dev))) return st;
    return launched(launch_rmsnorm_q8_1(x, gamma, B, K, eps, out, (cudaStream_t)stream),
                    "zq_rmsnorm_q8_1 launch");
}

int zq_q4k_gemv(const void *W, int N, int K, zq_q8_1 a, float *y, void *stream)
{
    int st = check_q4k(W, N, K, "zq_q4k_gemv");
    if (st) return st;
    if ((st = check_q8(a, "zq_q4k_gemv"))) return st;
    if (!y) return fail(ZQ_ERR_ARG, "zq_q4k_gemv: null y");
    if (!aligned16(y)) return fail(ZQ_ERR_ALIGN, "zq_q4k_gemv: y must be 16-byte aligned");
    int dev;
    if ((st = check_device(&dev))) return st;
    return launched(launch_gemv_dispatch(W, nullptr, N, K, a, y, nullptr, (cudaStream_t)stream),
                    "zq_q4k_gemv launch");
}

int zq_q4k_gemv_pair(const void *Wg, const void *Wu, int N, int K, zq_q8_1 a, float *y_gate,
                     float *y_up, void *stream)
{
    int st = check_q4k(Wg, N, K, "zq_q4k_gemv_pair (gate)");
    if (st) return st;
    if ((st = check_q4k(Wu, N, K, "zq_q4k_gemv_pair (up)"))) return st;
    if ((st = check_q8(a, "zq_q4k_gemv_pair"))) return st;
    if (!y_gate || !y_up) return fail(ZQ_ERR_ARG, "zq_q4k_gemv_pair: null output");
    if (!aligned16(y_gate) || !aligned16(y_up))
        return fail(ZQ_ERR_ALIGN, "zq_q4k_gemv_pair: outputs must be 16-byte aligned");
    int dev;
    if ((st = check_device(&dev))) return st;
    return launched(launch_gemv_dispatch(Wg, Wu, N, K, a, y_gate, y_up, (cudaStream_t)stream),
                    "zq_q4k_gemv_pair launch");
}

}  // extern "C"

namespace {

// Checks shared by the multi-matrix decode entry points; fills the job.
int check_job(const char *name, int nmat, const void *const *W, const int *N, int K, float *const *y, GemvJob &job)
{
    if (nmat < 1 || nmat > kGemvMaxMats)
        return fail(ZQ_ERR_ARG, "%s: nmat = %d must be in [1, %d]", name, nmat, kGemvMaxMats);
    if (!W || !N || !y) return fail(ZQ_ERR_ARG, "%s: null W, N or y array", name);
    job = GemvJob{};
    job.nmat = nmat;
    for (int m = 0; m < nmat; ++m) {
        int st = check_q4k(W[m], N[m], K, name);
        if (st) return st;
        if (!y[m]) return fail(ZQ_ERR_ARG, "%s: null y[%d]", name, m);
        if (!aligned16(y[m])) return fail(ZQ_ERR_ALIGN, "%s: y[%d] must be 16-byte aligned", name, m);
        job.W[m] = W[m];
        job.N[m] = N[m];
        job.y[m] = y[m];
    }
    return ZQ_OK;
}

}  // namespace

extern "C" {

int zq_q4k_gemv_multi(int nmat, const void *const *W, const int *N, int K, zq_q8_1 a, float *const *y,
                      void *stream)
{
    GemvJob job;
    int st = check_job("zq_q4k_gemv_multi", nmat, W, N, K, y, job);
    if (st) return st;
    if ((st = check_q8(a, "zq_q4k_gemv_multi"))) return st;
    int dev;
    if ((st = check_device(&dev))) return st;
    cudaStream_t s = (cudaStream_t)stream;
    if (gemv_stream_supported(K)) return launched(launch_gemv_stream(job, K, a, s), "zq_q4k_gemv_multi launch");
    for (int m = 0; m < nmat; ++m) {   // wide rows: one direct-load launch per matrix
        cudaError_t e = launch_gemv(job.W[m], nullptr, job.N[m], K, a, 1, job.y[m], nullptr, nullptr, s);
        if (e != cudaSuccess) return launched(e, "zq_q4k_gemv_multi launch");
    }
    return ZQ_OK;
}

int zq_rmsnorm_q4k_gemv(const float *x, const float *gamma, float eps, int K, int nmat, const void *const *W,
                        const int *N, float *const *y, const zq_q8_1 *q8_out, const void *l2_prefetch,
                        size_t l2_prefetch_bytes, void *stream)
{
    if (!x || !gamma) return fail(ZQ_ERR_ARG, "zq_rmsnorm_q4k_gemv: null x or gamma");
    if (!aligned16(x) || !aligned16(gamma))
        return fail(ZQ_ERR_ALIGN, "zq_rmsnorm_q4k_gemv: x and gamma must be 16-byte aligned");
    if (!(eps >= 0.0f) || eps != eps) return fail(ZQ_ERR_ARG, "zq_rmsnorm_q4k_gemv: eps must be >= 0");
    GemvJob job;
    int st = check_job("zq_rmsnorm_q4k_gemv", nmat, W, N, K, y, job);
    if (st) return st;
    if (!gemv_stream_supported(K))
        return fail(ZQ_ERR_SHAPE, "zq_rmsnorm_q4k_gemv: K = %d above the in-kernel normalisation limit 32768", K);
    if (q8_out && (st = check_q8(*q8_out, "zq_rmsnorm_q4k_gemv (q8_out)"))) return st;
    if (l2_prefetch && !aligned16(l2_prefetch))
        return fail(ZQ_ERR_ALIGN, "zq_rmsnorm_q4k_gemv: l2_prefetch must be 16-byte aligned");
    int dev;
    if ((st = check_device(&dev))) return st;
    return launched(launch_gemv_stream_fused(job, K, x, gamma, eps, false, q8_out, l2_prefetch,
                                             l2_prefetch ? l2_prefetch_bytes : 0, (cudaStream_t)stream),
                    "zq_rmsnorm_q4k_gemv launch");
}

int zq_rmsnorm_q4k_gemm(const float *x, const float *gamma, float eps, int B, int K, const void *W, int N, float *y,
                        const zq_q8_1 *q8_out, void *workspace, size_t workspace_bytes, void *stream)
{
    const char *name = "zq_rmsnorm_q4k_gemm";
    if (!x || !gamma || !y) return fail(ZQ_ERR_ARG, "%s: null x, gamma or y", name);
    if (!aligned16(x) || !aligned16(gamma) || !aligned16(y))
        return fail(ZQ_ERR_ALIGN, "%s: x, gamma and y must be 16-byte aligned", name);
    if (!(eps >= 0.0f) || eps != eps) return fail(ZQ_ERR_ARG, "%s: eps must be >= 0", name);
    int st = check_q4k(W, N, K, name);
    if (st) return st;
    if (K > 32768) return fail(ZQ_ERR_SHAPE, "%s: K = %d above the in-kernel normalisation limit 32768", name, K);
    if (B < 1 || B > 65536) return fail(ZQ_ERR_SHAPE, "%s: B = %d must be in [1, 65536]", name, B);
    if (q8_out && (st = check_q8(*q8_out, name))) return st;
    const bool streamed = B > 1 && chunk_streams(B, K);
    if (streamed && !q8_out) return fail(ZQ_ERR_ARG, "%s: B = %d needs q8_out (the codes the mat-vec reads)", name, B);
    const size_t need = (B == 1 || streamed) ? 0 : gemm_tc_workspace_bytes(N, K, B);
    if (need && (!workspace || workspace_bytes < need))
        return fail(ZQ_ERR_WORKSPACE, "%s: workspace of %zu bytes required, got %zu", name, need,
                    workspace ? workspace_bytes : (size_t)0);
    if (need && !aligned16(workspace)) return fail(ZQ_ERR_ALIGN, "%s: workspace must be 16-byte aligned", name);
    int dev;
    if ((st = check_device(&dev))) return st;
    cudaStream_t s = (cudaStream_t)stream;
    if (B == 1) {
        GemvJob job{};
        job.nmat = 1;
        job.W[0] = W;
        job.N[0] = N;
        job.y[0] = y;
        return launched(launch_gemv_stream_fused(job, K, x, gamma, eps, false, q8_out, nullptr, 0, s), name);
    }
    cudaError_t e;
    if (streamed) {
        if ((e = launch_rmsnorm_q8_1(x, gamma, B, K, eps, *q8_out, s)) != cudaSuccess) return launched(e, name);
        return launched(launch_q4k_tokens(W, N, K, *q8_out, B, y, s), name);
    }
    const TcWorkspace w = tc_workspace(workspace, K, B);
    if ((e = launch_rmsnorm_q8_1_split(x, gamma, B, K, eps, q8_out, w.hi, w.lo, w.tscale, w.s8x, s)) != cudaSuccess)
        return launched(e, name);
    return launched(launch_gemm_tc_split_done(W, N, K, B, y, workspace, true, s), name);
}

size_t zq_q4k_gemm_workspace_bytes(int N, int K, int B)
{
    if (N < 1 || K < 256 || K % 256 || B < 1) return 0;
    return chunk_streams(B, K) ? 0 : gemm_tc_workspace_bytes(N, K, B);
}

int zq_q4k_gemm(const void *W, int N, int K, zq_q8_1 a, int B, float *y, void *workspace,
                size_t workspace_bytes, void *stream)
{
    int st = check_q4k(W, N, K, "zq_q4k_gemm");
    if (st) return st;
    if ((st = check_q8(a, "zq_q4k_gemm"))) return st;
    if (B < 1 || B > 65536) return fail(ZQ_ERR_SHAPE, "zq_q4k_gemm: B = %d must be in [1, 65536]", B);
    if (!y) return fail(ZQ_ERR_ARG, "zq_q4k_gemm: null y");
    if (!aligned16(y)) return fail(ZQ_ERR_ALIGN, "zq_q4k_gemm: y must be 16-byte aligned");
    const size_t need = chunk_streams(B, K) ? 0 : gemm_tc_workspace_bytes(N, K, B);
    if (need && (!workspace || workspace_bytes < need))
        return fail(ZQ_ERR_WORKSPACE, "zq_q4k_gemm: workspace of %zu bytes required, got %zu", need,
                    workspace ? workspace_bytes : (size_t)0);
    if (need && !aligned16(workspace))
        return fail(ZQ_ERR_ALIGN, "zq_q4k_gemm: workspace must be 16-byte aligned");
    int dev;
    if ((st = check_device(&dev))) return st;
    cudaStream_t s = (cudaStream_t)stream;
    if (B == 1) return launched(launch_gemv_dispatch(W, nullptr, N, K, a, y, nullptr, s), "zq_q4k_gemm (B=1)");
    if (chunk_streams(B, K)) return launched(launch_q4k_tokens(W, N, K, a, B, y, s), "zq_q4k_gemm (B<=4)");
    return launched(launch_gemm_tc(W, N, K, a, B, y, workspace, true, s),
                    B <= 16 ? "zq_q4k_gemm (chunk)" : "zq_q4k_gemm (prefill)");
}

int zq_q4k_gemm_noalloc(const void *W, int N, int K, zq_q8_1 a, int B, float *y, void *stream)
{
    int st = check_q4k(W, N, K, "zq_q4k_gemm_noalloc");
    if (st) return st;
    if ((st = check_q8(a, "zq_q4k_gemm_noalloc"))) return st;
    if (B < 1 || B > 65536) return fail(ZQ_ERR_SHAPE, "zq_q4k_gemm_noalloc: B = %d must be in [1, 65536]", B);
    if (!y) return fail(ZQ_ERR_ARG, "zq_q4k_gemm_noalloc: null y");
    if (!aligned16(y)) return fail(ZQ_ERR_ALIGN, "zq_q4k_gemm_noalloc: y must be 16-byte aligned");
    const size_t need = chunk_streams(B, K) ? 0 : gemm_tc_workspace_bytes(N, K, B, false);
    if (need > noalloc_scratch_bytes())
        return fail(ZQ_ERR_WORKSPACE,
                    "zq_q4k_gemm_noalloc: B*K = %lld needs %zu bytes of scratch, more than the built-in %zu "
                    "(B*K <= 10485760); use zq_q4k_gemm with a workspace",
                    (long long)B * K, need, noalloc_scratch_bytes());
    int dev;
    if ((st = check_device(&dev))) return st;
    cudaStream_t s = (cudaStream_t)stream;
    if (B == 1) return launched(launch_gemv_dispatch(W, nullptr, N, K, a, y, nullptr, s), "zq_q4k_gemm_noalloc (B=1)");
    if (chunk_streams(B, K)) return launched(launch_q4k_tokens(W, N, K, a, B, y, s), "zq_q4k_gemm_noalloc (B<=4)");
    return launched(launch_gemm_noalloc(W, N, K, a, B, y, s), "zq_q4k_gemm_noalloc");
}

int zq_silu_mul_q8_1(const float *gate, const float *up, int B, int K, zq_q8_1 out, void *stream)
{
    if (!gate || !up) return fail(ZQ_ERR_ARG, "zq_silu_mul_q8_1: null gate or up");
    if (!aligned16(gate) || !aligned16(up))
        return fail(ZQ_ERR_ALIGN, "zq_silu_mul_q8_1: gate and up must be 16-byte aligned");
    if (B < 1 || B > 65535) return fail(ZQ_ERR_SHAPE, "zq_silu_mul_q8_1: B = %d out of range", B);
    if (K < 32 || K % 32 != 0 || K > (1 << 22))
        return fail(ZQ_ERR_SHAPE, "zq_silu_mul_q8_1: K = %d must be a multiple of 32 in [32, 2^22]", K);
    int st = check_q8(out, "zq_silu_mul_q8_1");
    if (st) return st;
    int dev;
    if ((st = check_device(&dev))) return st;
    return launched(launch_silu_mul_q8_1(gate, up, B, K, out, (cudaStream_t)stream), "zq_silu_mul_q8_1 launch");
}

int zq_silu_q4k_gemv(const float *gate, const float *up, int K, int nmat, const void *const *W, const int *N,
                     float *const *y, const zq_q8_1 *q8_out, const void *l2_prefetch, size_t l2_prefetch_bytes,
                     void *stream)
{
    if (!gate || !up) return fail(ZQ_ERR_ARG, "zq_silu_q4k_gemv: null gate or up");
    if (!aligned16(gate) || !aligned16(up))
        return fail(ZQ_ERR_ALIGN, "zq_silu_q4k_gemv: gate and up must be 16-byte aligned");
    GemvJob job;
    int st = check_job("zq_silu_q4k_gemv", nmat, W, N, K, y, job);
    if (st) return st;
    if (!gemv_stream_supported(K))
        return fail(ZQ_ERR_SHAPE, "zq_silu_q4k_gemv: K = %d above the in-kernel packing limit 32768", K);
    if (q8_out && (st = check_q8(*q8_out, "zq_silu_q4k_gemv (q8_out)"))) return st;
    if (l2_prefetch && !aligned16(l2_prefetch))
        return fail(ZQ_ERR_ALIGN, "zq_silu_q4k_gemv: l2_prefetch must be 16-byte aligned");
    int dev;
    if ((st = check_device(&dev))) return st;
    return launched(launch_gemv_stream_fused(job, K, gate, up, 0.0f, true, q8_out, l2_prefetch,
                                             l2_prefetch ? l2_prefetch_bytes : 0, (cudaStream_t)stream),
                    "zq_silu_q4k_gemv launch");
}

int zq_q4k_dequant_f16(const void *W, int N, int K, void *out, void *stream)
{
    int st = check_q4k(W, N, K, "zq_q4k_dequant_f16");
    if (st) return st;
    if (!out) return fail(ZQ_ERR_ARG, "zq_q4k_dequant_f16: null out");
    if (!aligned16(out)) return fail(ZQ_ERR_ALIGN, "zq_q4k_dequant_f16: out must be 16-byte aligned");
    int dev;
    if ((st = check_device(&dev))) return st;
    return launched(launch_q4k_dequant_f16(W, N, K, out, (cudaStream_t)stream), "zq_q4k_dequant_f16 launch");
}

int zq_q8_1_dequant_f16(zq_q8_1 a, int B, int K, void *out, void *stream)
{
    int st = check_q8(a, "zq_q8_1_dequant_f16");
    if (st) return st;
    if (B < 1 || K < 32 || K % 32) return fail(ZQ_ERR_SHAPE, "zq_q8_1_dequant_f16: B = %d, K = %d", B, K);
    if (!out) return fail(ZQ_ERR_ARG, "zq_q8_1_dequant_f16: null out");
    if (!aligned16(out)) return fail(ZQ_ERR_ALIGN, "zq_q8_1_dequant_f16: out must be 16-byte aligned");
    int dev;
    if ((st = check_device(&dev))) return st;
    return launched(launch_q8_1_dequant_f16(a, B, K, out, (cudaStream_t)stream), "zq_q8_1_dequant_f16 launch");
}

size_t zq_f16_gemm_workspace_bytes(int N, int K, int B)
{
    if (N < 1 || K < 64 || K % 64 || B < 1) return 0;
    return f16_gemm_workspace_bytes(N, K, B);
}

int zq_f16_gemm(const void *W16, int N, int K, const void *X16, int B, float *y, void *workspace,
                size_t workspace_bytes, void *stream)
{
    const char *name = "zq_f16_gemm";
    if (!W16 || !X16 || !y) return fail(ZQ_ERR_ARG, "%s: null pointer", name);
    if (!aligned16(W16) || !aligned16(X16) || !aligned16(y))
        return fail(ZQ_ERR_ALIGN, "%s: W16, X16 and y must be 16-byte aligned", name);
    if (N < 1 || B < 1 || B > 65536 || K < 64 || K % 64 || K > (1 << 20))
        return fail(ZQ_ERR_SHAPE, "%s: N = %d, K = %d, B = %d out of range", name, N, K, B);
    const size_t need = f16_gemm_workspace_bytes(N, K, B);
    if (need && (!workspace || workspace_bytes < need))
        return fail(ZQ_ERR_WORKSPACE, "%s: workspace of %zu bytes required, got %zu", name, need,
                    workspace ? workspace_bytes : (size_t)0);
    if (need && !aligned16(workspace)) return fail(ZQ_ERR_ALIGN, "%s: workspace must be 16-byte aligned", name);
    int dev, st;
    if ((st = check_device(&dev))) return st;
    return launched(launch_f16_gemm(W16, N, K, X16, B, y, static_cast<float *>(workspace), (cudaStream_t)stream),
                    name);
}

size_t zq_q5k_bytes(int N, int K)
{
    if (N < 1 || K < 256 || K % 256) return 0;
    return (size_t)N * (size_t)(K / 256) * 176;
}

size_t zq_q6k_bytes(int N, int K)
{
    if (N < 1 || K < 256 || K % 256) return 0;
    return (size_t)N * (size_t)(K / 256) * 210;
}

}  // extern "C"

namespace {

// Q5_K / Q6_K projection of B tokens (shared checks and dispatch).
int kq_gemm(bool q6, const char *name, const void *W, int N, int K, zq_q8_1 a, int B, float *y, void *stream)
{
    int st = check_q4k(W, N, K, name);
    if (st) return st;
    if (K > 32768) return fail(ZQ_ERR_SHAPE, "%s: K = %d above the staged-activation limit 32768", name, K);
    if ((st = check_q8(a, name))) return st;
    if (B < 1 || B > 16) return fail(ZQ_ERR_SHAPE, "%s: B = %d must be in [1, 16]", name, B);
    if (!y) return fail(ZQ_ERR_ARG, "%s: null y", name);
    if (!aligned16(y)) return fail(ZQ_ERR_ALIGN, "%s: y must be 16-byte aligned", name);
    int dev;
    if ((st = check_device(&dev))) return st;
    cudaStream_t s = (cudaStream_t)stream;
    return launched(q6 ? launch_q6k_tokens(W, N, K, a, B, y, s) : launch_q5k_tokens(W, N, K, a, B, y, s), name);
}

}  // namespace

extern "C" {

int zq_q5k_gemm(const void *W, int N, int K, zq_q8_1 a, int B, float *y, void *stream)
{
    return kq_gemm(false, "zq_q5k_gemm", W, N, K, a, B, y, stream);
}

int zq_q6k_gemm(const void *W, int N, int K, zq_q8_1 a, int B, float *y, void *stream)
{
    return kq_gemm(true, "zq_q6k_gemm", W, N, K, a, B, y, stream);
}

int zq_q5k_gemv(const void *W, int N, int K, zq_q8_1 a, float *y, void *stream)
{
    return kq_gemm(false, "zq_q5k_gemv", W, N, K, a, 1, y, stream);
}

int zq_q6k_gemv(const void *W, int N, int K, zq_q8_1 a, float *y, void *stream)
{
    return kq_gemm(true, "zq_q6k_gemv", W, N, K, a, 1, y, stream);
}

int zq_rmsnorm_q6k_gemv(const float *x, const float *gamma, float eps, int K, const void *W, int N, float *y,
                        const zq_q8_1 *q8_out, void *stream)
{
    const char *name = "zq_rmsnorm_q6k_gemv";
    if (!x || !gamma) return fail(ZQ_ERR_ARG, "%s: null x or gamma", name);
    if (!aligned16(x) || !aligned16(gamma)) return fail(ZQ_ERR_ALIGN, "%s: x and gamma must be 16-byte aligned", name);
    if (!(eps >= 0.0f) || eps != eps) return fail(ZQ_ERR_ARG, "%s: eps must be >= 0", name);
    GemvJob job;
    float *ys[1] = {y};
    int st = check_job(name, 1, &W, &N, K, ys, job);
    if (st) return st;
    if (K > 32768) return fail(ZQ_ERR_SHAPE, "%s: K = %d above the in-kernel normalisation limit 32768", name, K);
    if (q8_out && (st = check_q8(*q8_out, "zq_rmsnorm_q6k_gemv (q8_out)"))) return st;
    int dev;
    if ((st = check_device(&dev))) return st;
    return launched(launch_q6k_fused(job, K, x, gamma, eps, q8_out, (cudaStream_t)stream), name);
}

int zq_debug_stream_plan(int wtype, int ntok, int K, long long total_rows, int sms, int32_t *out)
{
    if (!out) return fail(ZQ_ERR_ARG, "zq_debug_stream_plan: null out");
    if (wtype < 4 || wtype > 6 || (ntok != 1 && ntok != 4))
        return fail(ZQ_ERR_ARG, "zq_debug_stream_plan: wtype %d / ntok %d unknown", wtype, ntok);
    if (K < 256 || K % 256 || K > 32768 || total_rows < 1 || sms < 1)
        return fail(ZQ_ERR_SHAPE, "zq_debug_stream_plan: K = %d, rows = %lld, sms = %d out of range", K, total_rows, sms);
    if (!stream_plan_query(wtype, ntok, K, total_rows, sms, out))
        return fail(ZQ_ERR_SHAPE, "zq_debug_stream_plan: the staging of %d token(s) of K = %d does not fit", ntok, K);
    return ZQ_OK;
}

int zq_debug_peak_probe(int kind, int blocks, int iters, void *sink, void *stream)
{
    if (kind < 0 || kind > 10) return fail(ZQ_ERR_ARG, "zq_debug_peak_probe: kind %d unknown", kind);
    if ((kind == 7 || kind >= 9) && blocks < 2)
        return fail(ZQ_ERR_SHAPE, "zq_debug_peak_probe: kinds 7, 9 and 10 need blocks >= 2");
    if (!sink || !aligned16(sink)) return fail(ZQ_ERR_ARG, "zq_debug_peak_probe: sink null or misaligned");
    if (blocks < 1 || blocks > 65535 || iters < 1 || iters > (1 << 24))
        return fail(ZQ_ERR_SHAPE, "zq_debug_peak_probe: blocks = %d, iters = %d out of range", blocks, iters);
    int dev, st;
    if ((st = check_device(&dev))) return st;
    return launched(launch_peak_probe(kind, blocks, iters, static_cast<int *>(sink), (cudaStream_t)stream),
                    "zq_debug_peak_probe");
}

int zq_debug_wait_expiry(const void *W, int N, int K, zq_q8_1 a, float *y, int withhold_stage,
                         unsigned int wait_us, int ctas, void *stream)
{
    const char *name = "zq_debug_wait_expiry";
    int st = check_q4k(W, N, K, name);
    if (st) return st;
    if ((st = check_q8(a, name))) return st;
    if (!y) return fail(ZQ_ERR_ARG, "%s: null y", name);
    if (K > 32768) return fail(ZQ_ERR_SHAPE, "%s: K = %d above 32768", name, K);
    if (withhold_stage < 0 || wait_us < 1 || wait_us > 2000000u)
        return fail(ZQ_ERR_ARG, "%s: withhold_stage = %d, wait_us = %u out of range", name, withhold_stage, wait_us);
    int dev;
    if ((st = check_device(&dev))) return st;
    if (ctas < 1 || ctas > num_sms())
        return fail(ZQ_ERR_ARG, "%s: ctas = %d out of range 1..%d", name, ctas, num_sms());
    return launched(launch_q4k_wait_expiry(W, N, K, a, y, withhold_stage, (uint64_t)wait_us * 1000u, ctas,
                                           (cudaStream_t)stream),
                    name);
}

int zq_device_status(unsigned int *flags, int clear)
{
    if (!flags) return fail(ZQ_ERR_ARG, "zq_device_status: null flags");
    int dev, st;
    if ((st = check_device(&dev))) return st;
    cudaError_t e = cudaMemcpyFromSymbol(flags, g_zq_device_status, sizeof(unsigned int));
    if (e == cudaSuccess && clear) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_zq_device_status, &zero, sizeof zero);
    }
    return launched(e, "zq_device_status");
}

int zq_copy(void *dst, const void *src, size_t bytes, void *stream)
{
    if (bytes == 0) return ZQ_OK;
    if (!dst || !src) return fail(ZQ_ERR_ARG, "zq_copy: null pointer");
    int dev, st;
    if ((st = check_device(&dev))) return st;
    void *d = nullptr, *s = nullptr;
    if ((st = device_address(dst, dev, &d, "zq_copy: dst"))) return st;
    if ((st = device_address(src, dev, &s, "zq_copy: src"))) return st;
    return launched(launch_copy(d, s, bytes, g_sms[dev], (cudaStream_t)stream), "zq_copy");
}

int zq_debug_q4k_isums(const void *W, int N, int K, zq_q8_1 a, int B, int32_t *isums, int path,
                       void *workspace, size_t workspace_bytes, void *stream)
{
    int st = check_q4k(W, N, K, "zq_debug_q4k_isums");
    if (st) return st;
    if ((st = check_q8(a, "zq_debug_q4k_isums"))) return st;
    if (B < 1 || B > 65536) return fail(ZQ_ERR_SHAPE, "zq_debug_q4k_isums: B = %d out of range", B);
    if (!isums || !aligned16(isums)) return fail(ZQ_ERR_ARG, "zq_debug_q4k_isums: isums null or misaligned");
    if (path < 0 || path > 2) return fail(ZQ_ERR_ARG, "zq_debug_q4k_isums: path %d unknown", path);
    if (path == 1 && B < 17) return fail(ZQ_ERR_SHAPE, "zq_debug_q4k_isums: path 1 needs B >= 17");
    if (path == 2 && (B < 2 || B > 16)) return fail(ZQ_ERR_SHAPE, "zq_debug_q4k_isums: path 2 needs 2 <= B <= 16");
    if (path != 0) {
        const size_t need = (size_t)2 * B * K;   // the binary16 copy of the activation codes
        if (need && (!workspace || workspace_bytes < need))
            return fail(ZQ_ERR_WORKSPACE, "zq_debug_q4k_isums: workspace of %zu bytes required", need);
    }
    int dev;
    if ((st = check_device(&dev))) return st;
    cudaStream_t s = (cudaStream_t)stream;
    if (path == 0) return launched(launch_gemv(W, nullptr, N, K, a, B, nullptr, nullptr, isums, s), "isums (dp4a)");
    return launched(launch_isums_tc(W, N, K, a, B, isums, workspace, s),
                    path == 1 ? "isums (tensor cores, prefill sizes)" : "isums (tensor cores, chunk sizes)");
}

}  // extern "C"
