// noalloc.cu -- q4_0_gemm_noalloc: the tensor-core GEMM without any device
// allocation.
//
// Why it exists.  q4_0_gemm needs scratch for the binary16 copy of x, which
// q4_0_matmul takes with cudaMallocAsync and q4_0_matmul_ws takes from the
// caller.  Some callers can do neither: code that runs where the CUDA
// allocator must not be entered (a host callback, a real-time loop that was
// promised no allocation after start-up, a plug-in whose host owns every
// device byte and hands it no workspace).  For them the scratch lives here,
// in a fixed array in device memory that this library reserves when it is
// loaded on a GPU and keeps until the process exits.
//
// Rules of use.
//   * The array holds Q4_0_NOALLOC_SCRATCH_BYTES (32 MiB): x of M rows and
//     K columns needs M * K * 2 bytes, so M * K <= 16 Mi elements (e.g.
//     M = 2048 at K = 5120, M = 512 at K = 17408).  Larger calls are refused
//     with Q4_0_ERR_WORKSPACE before anything is launched.
//   * The array is shared by every call on a device.  Calls whose kernels
//     overlap on the GPU (different streams without ordering between them)
//     race on it and give wrong results; order them on one stream.
//   * The first call on each device looks up the array's device address
//     (cudaGetSymbolAddress, with that device current).  Make that first call
//     before any stream capture begins.
//   * Each call overwrites the part of the array it uses before reading it,
//     so nothing needs to start at zero.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/q4_0.h"
#include "q4_0_internal.h"

namespace {

// The scratch itself.  In host code this name is only a stand-in for the
// device array: its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[Q4_0_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices];  // device address of the array, per device

// Device address of the array on the current device (looked up once per
// device, with that device current).  Returns nullptr on failure.
void *scratch_for_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
        g_scratch_ptr[dev] = p;
    }
    return g_scratch_ptr[dev];
}

}  // namespace

extern "C" int q4_0_gemm_noalloc(const uint16_t *x, const uint8_t *wq, float *y, int64_t M,
                                 int64_t N, int64_t K, void *stream) {
    // the same checks, in the same order, as q4_0_gemm
    const int st = q4_0::check_matmul_args(x, wq, y, M, N, K);
    if (st != Q4_0_OK) return st;
    if (!q4_0::gemm_shape_supported(M, N, K)) return Q4_0_ERR_UNSUPPORTED;
    if (M * K > (int64_t)(Q4_0_NOALLOC_SCRATCH_BYTES / 2) ||
        q4_0::gemm_workspace_bytes(M, N, K, 1) > Q4_0_NOALLOC_SCRATCH_BYTES)
        return Q4_0_ERR_WORKSPACE;
    void *scratch = scratch_for_current_device();
    if (!scratch) return Q4_0_ERR_CUDA;
    unsigned int *err = q4_0::device_error_word();
    if (!err) return Q4_0_ERR_CUDA;
    // K is never split here: the array holds the binary16 copy of x only
    const cudaError_t e =
        q4_0::launch_gemm(x, wq, y, false, M, N, K, scratch, 1, static_cast<cudaStream_t>(stream), err);
    return e == cudaSuccess ? Q4_0_OK : Q4_0_ERR_CUDA;
}
