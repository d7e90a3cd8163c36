// api.cu -- the C ABI of libq4_0.so (declared in include/q4_0.h): argument
// validation, the M-based dispatch between the decode GEMV and the tcgen05
// GEMM, scratch handling and the device error word.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "../../include/q4_0.h"
#include "q4_0_internal.h"
#include "q4_0_ptx.cuh"

namespace q4_0 {

// Written by a kernel that abandons a bounded wait; read and cleared by
// q4_0_device_error().
__device__ unsigned int g_device_error_word;

namespace {

// x from page-locked host memory into the workspace, for the decode kernels
// (M <= 2), whose every CTA reads all of x: read in place, a matmul of 152
// CTAs pulled 152 copies of x over the host link, on the critical path after
// its dependency wait.  x is read only after this kernel's own dependency
// wait: an earlier kernel on the stream may write it (y of an earlier call
// passed as x), and this library's kernels let their dependents start early.
__global__ void __launch_bounds__(256) stage_x_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst,
                                                      int64_t n16) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n16) dst[i] = src[i];
}

// Self-check of the bounded-wait path: one thread waits on an mbarrier that
// nothing arrives on, gives up after `limit_ns`, records the timeout in the
// device error word and returns -- the same path every pipeline wait in this
// library takes.  No trap, no fault: the context stays usable.
__global__ void wait_timeout_selftest_kernel(unsigned long long limit_ns, unsigned int *err) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);
    mbar_fence_init();
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(&bar, 0)) {
        if (global_ns() - t0 > limit_ns) {
            atomicExch(err, kErrWaitTimeout);
            return;
        }
    }
}

constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];
std::atomic<unsigned int *> g_err_ptr[kMaxDevices];
}  // namespace

int device_sm_count(int device) {
    if (device < 0 || device >= kMaxDevices) return 0;
    int v = g_sm_count[device].load(std::memory_order_relaxed);
    if (v > 0) return v;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return 0;
    g_sm_count[device].store(v, std::memory_order_relaxed);
    return v;
}

cudaError_t ensure_smem_attr(const void *func, int bytes) {
    struct Entry {
        const void *func;
        int device;
        int bytes;
    };
    static std::mutex mu;
    static Entry done[256];
    static int ndone = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < ndone; ++i)
        if (done[i].func == func && done[i].device == dev && done[i].bytes >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    for (int i = 0; i < ndone; ++i)
        if (done[i].func == func && done[i].device == dev) {
            done[i].bytes = bytes;
            return cudaSuccess;
        }
    if (ndone < 256) done[ndone++] = Entry{func, dev, bytes};
    return cudaSuccess;
}

unsigned int *device_error_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    unsigned int *p = g_err_ptr[dev].load(std::memory_order_acquire);
    if (p) return p;
    void *addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_device_error_word) != cudaSuccess) return nullptr;
    p = static_cast<unsigned int *>(addr);
    g_err_ptr[dev].store(p, std::memory_order_release);
    return p;
}

}  // namespace q4_0

using namespace q4_0;

namespace {
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
}  // namespace

namespace q4_0 {
// Common validation of a matmul call.
// `any_k`: K % 32 == 0 is enough (the dispatcher pads other K to a multiple
// of 256); the kernel-alone entry points need K % 256 == 0.
int check_matmul_args(const void *x, const void *wq, const void *y, int64_t M, int64_t N,
                      int64_t K, bool any_k) {
    if (!x || !wq || !y) return Q4_0_ERR_INVALID_ARG;
    if (M < 1 || N < 1 || K < 32 || K % 32 != 0) return Q4_0_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(wq) || !aligned16(y)) return Q4_0_ERR_INVALID_ARG;
    if (K % 256 != 0 && !any_k) return Q4_0_ERR_UNSUPPORTED;
    // keep every index and TMA coordinate in 32-bit range
    if (M > (1ll << 30) || N > (1ll << 30) || K > (1ll << 24)) return Q4_0_ERR_UNSUPPORTED;
    if (M * K > (1ll << 40) || N * K > (1ll << 40) || M * N > (1ll << 40))
        return Q4_0_ERR_UNSUPPORTED;
    return Q4_0_OK;
}
}  // namespace q4_0

namespace {

int from_cuda(cudaError_t e) { return e == cudaSuccess ? Q4_0_OK : Q4_0_ERR_CUDA; }

// The device address of page-locked host memory the current device can
// access, or nullptr (pageable or unknown memory, or a query error).
const void *host_mapping(const void *p) {
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
}

}  // namespace

extern "C" {

int q4_0_version(void) { return Q4_0_VERSION; }

const char *q4_0_status_string(int status) {
    switch (status) {
        case Q4_0_OK: return "ok";
        case Q4_0_ERR_INVALID_ARG: return "invalid argument";
        case Q4_0_ERR_UNSUPPORTED: return "unsupported by this build";
        case Q4_0_ERR_CUDA: return "CUDA error";
        case Q4_0_ERR_DEVICE_TIMEOUT: return "device wait timed out";
        case Q4_0_ERR_WORKSPACE: return "workspace missing or too small";
        default: return "unknown status";
    }
}

size_t q4_0_weight_bytes(int64_t N, int64_t K) {
    if (N < 1 || K < 1 || K % 32 != 0) return 0;
    return (size_t)N * (size_t)(K / 32) * Q4_0_BLOCK_BYTES;
}

int q4_0_quantize(const float *w, uint8_t *wq, int64_t N, int64_t K, void *stream) {
    if (!w || !wq || N < 1 || K < 32 || K % 32 != 0) return Q4_0_ERR_INVALID_ARG;
    if (!aligned16(w) || (reinterpret_cast<uintptr_t>(wq) & 1u)) return Q4_0_ERR_INVALID_ARG;
    if (N * (K / 32) > (1ll << 40)) return Q4_0_ERR_UNSUPPORTED;
    return from_cuda(launch_quantize(w, wq, N, K, static_cast<cudaStream_t>(stream),
                                     device_error_word()));
}

namespace {
// K split of the GEMM on the current device (1 when it cannot be queried).
int current_splits(int64_t M, int64_t N, int64_t K) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    return gemm_splits(M, N, K, device_sm_count(dev));
}
}  // namespace

size_t q4_0_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    if (M < 1 || N < 1 || K < 1) return 0;
    return gemm_workspace_bytes(M, N, K, current_splits(M, N, K));
}

int q4_0_gemm_plan(int64_t M, int64_t N, int64_t K, int *tile_rows, int *splits, int *persistent) {
    if (!tile_rows || !splits || !persistent || M < 1 || N < 1 || K < 256 || K % 256 != 0)
        return Q4_0_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return Q4_0_ERR_CUDA;
    const int sms = device_sm_count(dev);
    *splits = gemm_splits(M, N, K, sms);
    gemm_plan(M, N, K, sms, *splits, tile_rows, persistent);
    return Q4_0_OK;
}

size_t q4_0_gemv_workspace_bytes(int64_t M, int64_t K) {
    if (M < 1 || M > kGemvMaxM || K < 1) return 0;
    return gemv_workspace_bytes(M, K);
}

size_t q4_0_matmul_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    if (M < 1 || N < 1 || K < 32 || K % 32 != 0) return 0;
    // other K: the zero-padded copies of W and x, then the padded problem's own
    const size_t pad = pad_bytes(M, N, K);
    const int64_t kp = padded_k(K);
    if (M <= kDecodeMaxM) return pad + q4_0_gemv_workspace_bytes(M, kp);
    return pad + q4_0_gemm_workspace_bytes(M, N, kp);
}

namespace {
// The decode and GEMM paths with the output element type as a flag (the
// public entry points below are these with fp32 y, or q4_0_matmul_ex).
int gemv_ws_impl(const uint16_t *x, const uint8_t *wq, float *y, bool ybf16, int64_t M, int64_t N, int64_t K,
                 void *workspace, size_t workspace_bytes, void *stream) {
    int st = check_matmul_args(x, wq, y, M, N, K);
    if (st != Q4_0_OK) return st;
    if (M > kGemvMaxM || !gemv_shape_supported(M, N, K)) return Q4_0_ERR_UNSUPPORTED;
    const size_t need = gemv_workspace_bytes(M, K);
    if (need && (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u)))
        return Q4_0_ERR_WORKSPACE;
    unsigned int *err = device_error_word();
    if (!err) return Q4_0_ERR_CUDA;
    return from_cuda(launch_gemv(x, wq, y, ybf16, M, N, K, need ? workspace : nullptr,
                                 static_cast<cudaStream_t>(stream), err));
}

int gemm_impl(const uint16_t *x, const uint8_t *wq, float *y, bool ybf16, int64_t M, int64_t N, int64_t K,
              void *workspace, size_t workspace_bytes, void *stream) {
    int st = check_matmul_args(x, wq, y, M, N, K);
    if (st != Q4_0_OK) return st;
    if (!gemm_shape_supported(M, N, K)) return Q4_0_ERR_UNSUPPORTED;
    // split K only if the workspace has room for the partial tiles
    int splits = current_splits(M, N, K);
    if (workspace_bytes < gemm_workspace_bytes(M, N, K, splits)) splits = 1;
    if (!workspace || workspace_bytes < gemm_workspace_bytes(M, N, K, 1) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return Q4_0_ERR_WORKSPACE;
    unsigned int *err = device_error_word();
    if (!err) return Q4_0_ERR_CUDA;
    return from_cuda(
        launch_gemm(x, wq, y, ybf16, M, N, K, workspace, splits, static_cast<cudaStream_t>(stream), err));
}

int matmul_ws_impl(const uint16_t *x, const uint8_t *wq, float *y, bool ybf16, int64_t M, int64_t N, int64_t K,
                   void *workspace, size_t workspace_bytes, void *stream) {
    int st = check_matmul_args(x, wq, y, M, N, K, true);
    if (st != Q4_0_OK) return st;
    const int64_t kk = K % 256 != 0 ? padded_k(K) : K;
    if (M <= kDecodeMaxM ? !gemv_shape_supported(M, N, kk) : !gemm_shape_supported(M, N, kk))
        return Q4_0_ERR_UNSUPPORTED;
    if (K % 256 != 0) {
        // copy W and x, zero-padded to a multiple of 256, then run the padded problem
        const size_t pad = pad_bytes(M, N, K);
        if (!workspace || workspace_bytes < q4_0_matmul_workspace_bytes(M, N, K) ||
            (reinterpret_cast<uintptr_t>(workspace) & 255u))
            return Q4_0_ERR_WORKSPACE;
        uint16_t *xp = nullptr;
        uint8_t *wqp = nullptr;
        if (launch_pad(x, wq, M, N, K, workspace, &xp, &wqp, static_cast<cudaStream_t>(stream)) != cudaSuccess)
            return Q4_0_ERR_CUDA;
        void *rest = static_cast<uint8_t *>(workspace) + pad;
        const size_t rest_bytes = workspace_bytes - pad;
        const int64_t kp = padded_k(K);
        if (M <= kDecodeMaxM)
            return gemv_ws_impl(xp, wqp, y, ybf16, M, N, kp, rest_bytes ? rest : nullptr, rest_bytes, stream);
        return gemm_impl(xp, wqp, y, ybf16, M, N, kp, rest, rest_bytes, stream);
    }
    if (M <= kDecodeMaxM) return gemv_ws_impl(x, wq, y, ybf16, M, N, K, workspace, workspace_bytes, stream);
    return gemm_impl(x, wq, y, ybf16, M, N, K, workspace, workspace_bytes, stream);
}

// As matmul_ws_impl with scratch taken by cudaMallocAsync on the stream.
int matmul_alloc_impl(const uint16_t *x, const uint8_t *wq, float *y, bool ybf16, int64_t M, int64_t N,
                      int64_t K, void *stream) {
    int st = check_matmul_args(x, wq, y, M, N, K, true);
    if (st != Q4_0_OK) return st;
    const size_t bytes = q4_0_matmul_workspace_bytes(M, N, K);
    if (bytes == 0) return matmul_ws_impl(x, wq, y, ybf16, M, N, K, nullptr, 0, stream);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void *ws = nullptr;
    if (cudaMallocAsync(&ws, bytes, s) != cudaSuccess) return Q4_0_ERR_CUDA;
    st = matmul_ws_impl(x, wq, y, ybf16, M, N, K, ws, bytes, stream);
    const cudaError_t fe = cudaFreeAsync(ws, s);
    if (st == Q4_0_OK && fe != cudaSuccess) st = Q4_0_ERR_CUDA;
    return st;
}
}  // namespace

int q4_0_gemv_ws(const uint16_t *x, const uint8_t *wq, float *y, int64_t M, int64_t N, int64_t K,
                 void *workspace, size_t workspace_bytes, void *stream) {
    return gemv_ws_impl(x, wq, y, false, M, N, K, workspace, workspace_bytes, stream);
}

int q4_0_gemv(const uint16_t *x, const uint8_t *wq, float *y, int64_t M, int64_t N, int64_t K,
              void *stream) {
    int st = check_matmul_args(x, wq, y, M, N, K);
    if (st != Q4_0_OK) return st;
    if (M > kGemvMaxM) return Q4_0_ERR_UNSUPPORTED;
    return matmul_alloc_impl(x, wq, y, false, M, N, K, stream);
}

int q4_0_gemm(const uint16_t *x, const uint8_t *wq, float *y, int64_t M, int64_t N, int64_t K,
              void *workspace, size_t workspace_bytes, void *stream) {
    return gemm_impl(x, wq, y, false, M, N, K, workspace, workspace_bytes, stream);
}

int q4_0_matmul_ws(const uint16_t *x, const uint8_t *wq, float *y, int64_t M, int64_t N, int64_t K,
                   void *workspace, size_t workspace_bytes, void *stream) {
    return matmul_ws_impl(x, wq, y, false, M, N, K, workspace, workspace_bytes, stream);
}

int q4_0_matmul(const uint16_t *x, const uint8_t *wq, float *y, int64_t M, int64_t N, int64_t K,
                void *stream) {
    return matmul_alloc_impl(x, wq, y, false, M, N, K, stream);
}

int q4_0_matmul_ex(const uint16_t *x, const uint8_t *wq, void *y, int y_type, int64_t M, int64_t N, int64_t K,
                   void *workspace, size_t workspace_bytes, void *stream) {
    if (y_type != Q4_0_Y_F32 && y_type != Q4_0_Y_BF16) return Q4_0_ERR_INVALID_ARG;
    float *yf = static_cast<float *>(y);
    const bool bf16 = y_type == Q4_0_Y_BF16;
    if (!workspace && workspace_bytes == 0 && q4_0_matmul_workspace_bytes(M, N, K) != 0)
        return matmul_alloc_impl(x, wq, yf, bf16, M, N, K, stream);
    return matmul_ws_impl(x, wq, yf, bf16, M, N, K, workspace, workspace_bytes, stream);
}

int q4_0_matmul_grouped(int G, const uint16_t *const *x, const uint8_t *const *wq, void *const *y, int y_type,
                        int64_t M, const int64_t *N, const int64_t *K, void *stream) {
    if (G < 0 || G > 4096) return Q4_0_ERR_INVALID_ARG;
    if (G == 0) return Q4_0_OK;
    if (!x || !wq || !y || !N || !K) return Q4_0_ERR_INVALID_ARG;
    if (y_type != Q4_0_Y_F32 && y_type != Q4_0_Y_BF16) return Q4_0_ERR_INVALID_ARG;
    // every problem is checked before anything is launched
    for (int g = 0; g < G; ++g) {
        const int st = check_matmul_args(x[g], wq[g], y[g], M, N[g], K[g], true);
        if (st != Q4_0_OK) return st;
        const int64_t kk = K[g] % 256 != 0 ? padded_k(K[g]) : K[g];
        if (M <= kDecodeMaxM ? !gemv_shape_supported(M, N[g], kk) : !gemm_shape_supported(M, N[g], kk))
            return Q4_0_ERR_UNSUPPORTED;
    }
    unsigned int *err = device_error_word();
    if (!err) return Q4_0_ERR_CUDA;
    const bool bf16 = y_type == Q4_0_Y_BF16;
    float *const *yf = reinterpret_cast<float *const *>(y);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // runs of problems the grouped decode takes go out together; any other
    // problem is one q4_0_matmul_ex call, in order
    for (int g = 0; g < G;) {
        int e = g;
        while (e < G && grouped_decode_eligible(M, N[e], K[e])) ++e;
        if (e > g) {
            const int st = from_cuda(launch_gemv_grouped(e - g, x + g, wq + g, yf + g, bf16, M, N + g, K + g, s, err));
            if (st != Q4_0_OK) return st;
            g = e;
            continue;
        }
        const int st = q4_0_matmul_ex(x[g], wq[g], y[g], y_type, M, N[g], K[g], nullptr, 0, stream);
        if (st != Q4_0_OK) return st;
        ++g;
    }
    return Q4_0_OK;
}

int q4_0_matmul_grouped_launches(int G, int64_t M, const int64_t *N, const int64_t *K) {
    if (G < 1 || G > 4096 || !N || !K) return -1;
    for (int g = 0; g < G; ++g)
        if (N[g] < 1 || K[g] < 32 || K[g] % 32 != 0 || !grouped_decode_eligible(M, N[g], K[g])) return -1;
    return grouped_decode_launches(G, M, N, K);
}

size_t q4_0_matmul_host_workspace_bytes(int64_t M, int64_t N, int64_t K, int y_type) {
    if (y_type != Q4_0_Y_F32 && y_type != Q4_0_Y_BF16) return 0;
    if (M < 1 || N < 1 || K < 32 || K % 32 != 0) return 0;
    if (M > (1ll << 30) || N > (1ll << 30) || K > (1ll << 24) || M * K > (1ll << 40) || M * N > (1ll << 40))
        return 0;
    const size_t ysz = y_type == Q4_0_Y_BF16 ? 2 : 4;
    const size_t xb = ((size_t)M * (size_t)K * 2 + 255) / 256 * 256;
    const size_t yb = ((size_t)M * (size_t)N * ysz + 255) / 256 * 256;
    return xb + yb + q4_0_matmul_workspace_bytes(M, N, K);
}

int q4_0_matmul_host(const uint16_t *x_host, const uint8_t *wq, void *y_host, int y_type, int64_t M, int64_t N,
                     int64_t K, void *workspace, size_t workspace_bytes, void *stream) {
    if (y_type != Q4_0_Y_F32 && y_type != Q4_0_Y_BF16) return Q4_0_ERR_INVALID_ARG;
    if (!x_host || !wq || !y_host) return Q4_0_ERR_INVALID_ARG;
    const size_t need = q4_0_matmul_host_workspace_bytes(M, N, K, y_type);
    if (need == 0) return Q4_0_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < need || !aligned16(workspace)) return Q4_0_ERR_WORKSPACE;
    const bool bf16 = y_type == Q4_0_Y_BF16;
    const size_t ysz = bf16 ? 2 : 4;
    const size_t xbytes = (size_t)M * (size_t)K * 2, ybytes = (size_t)M * (size_t)N * ysz;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    uint16_t *xd = reinterpret_cast<uint16_t *>(ws);
    uint8_t *yd = ws + (xbytes + 255) / 256 * 256;
    uint8_t *rest = yd + (ybytes + 255) / 256 * 256;
    const size_t rest_bytes = workspace_bytes - (size_t)(rest - ws);
    // Page-locked host memory that the device can address (on a GB300 the
    // Grace memory is coherent with the GPU over NVLink-C2C): the kernels
    // read x and write y there directly, so no copy stands between this call
    // and the previous one on the stream.  Other host memory is copied.
    const void *xdev = host_mapping(x_host), *ydev = host_mapping(y_host);
    if (xdev && ydev && aligned16(xdev) && aligned16(ydev)) {
        const size_t own = q4_0_matmul_workspace_bytes(M, N, K);
        const uint16_t *xk = static_cast<const uint16_t *>(xdev);
        if (M <= 2) {
            // the decode kernels read x in every CTA: one copy into the workspace first
            const int st = check_matmul_args(xk, wq, static_cast<const float *>(ydev), M, N, K, true);
            if (st != Q4_0_OK) return st;
            const int64_t n16 = (int64_t)(xbytes / 16);
            const cudaError_t e = launch_pdl(stage_x_kernel, dim3((unsigned)((n16 + 255) / 256)), dim3(256), 0,
                                             static_cast<cudaStream_t>(stream), reinterpret_cast<const uint4 *>(xk),
                                             reinterpret_cast<uint4 *>(xd), n16);
            if (e != cudaSuccess) return Q4_0_ERR_CUDA;
            xk = xd;
        }
        return matmul_ws_impl(xk, wq, static_cast<float *>(const_cast<void *>(ydev)), bf16, M, N, K,
                              own ? rest : nullptr, rest_bytes, stream);
    }
    int st = check_matmul_args(xd, wq, yd, M, N, K, true);
    if (st != Q4_0_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(xd, x_host, xbytes, cudaMemcpyHostToDevice, s) != cudaSuccess) return Q4_0_ERR_CUDA;
    st = matmul_ws_impl(xd, wq, reinterpret_cast<float *>(yd), bf16, M, N, K,
                        q4_0_matmul_workspace_bytes(M, N, K) ? rest : nullptr, rest_bytes, stream);
    if (st != Q4_0_OK) return st;
    return from_cuda(cudaMemcpyAsync(y_host, yd, ybytes, cudaMemcpyDeviceToHost, s));
}

int q4_0_selftest_wait_timeout(int64_t limit_us, void *stream) {
    if (limit_us < 1 || limit_us > 1000000) return Q4_0_ERR_INVALID_ARG;
    unsigned int *err = device_error_word();
    if (!err) return Q4_0_ERR_CUDA;
    wait_timeout_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        (unsigned long long)limit_us * 1000ull, err);
    return from_cuda(cudaGetLastError());
}

int q4_0_device_error(int *code) {
    if (!code) return Q4_0_ERR_INVALID_ARG;
    unsigned int v = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return Q4_0_ERR_CUDA;
    if (cudaMemcpyFromSymbol(&v, g_device_error_word, sizeof v) != cudaSuccess) return Q4_0_ERR_CUDA;
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_device_error_word, &zero, sizeof zero) != cudaSuccess)
        return Q4_0_ERR_CUDA;
    *code = v ? Q4_0_ERR_DEVICE_TIMEOUT : Q4_0_OK;
    return Q4_0_OK;
}

}  // extern "C"
