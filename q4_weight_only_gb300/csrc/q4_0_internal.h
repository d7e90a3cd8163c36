// q4_0_internal.h -- launchers shared between the translation units of
// libq4_0.so (not part of the public ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace q4_0 {

// Per-device facts, queried once per device.
int device_sm_count(int device);

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) once per (kernel, device),
// so that later launches (possibly inside a stream capture) only launch.
cudaError_t ensure_smem_attr(const void *func, int bytes);
// Launch with programmatic stream serialization allowed, so the kernel may
// begin while the previous kernel in the stream is still running (it must
// call griddepcontrol.wait before reading anything that kernel wrote).
template <typename... Params, typename... Actual>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Actual &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Actual &&>(args)...);
}

// Device error word of the current device (a __device__ variable's address).
unsigned int *device_error_word();

// Validation shared by every matmul entry point: a Q4_0 status code.
// `any_k`: K % 32 == 0 is enough (the dispatcher pads other K to a multiple
// of 256); the kernel-alone entry points need K % 256 == 0.
int check_matmul_args(const void *x, const void *wq, const void *y, int64_t M, int64_t N, int64_t K,
                      bool any_k = false);

cudaError_t launch_quantize(const float *w, uint8_t *wq, int64_t N, int64_t K, cudaStream_t s,
                            unsigned int *err);

// y is fp32, or bfloat16 when `ybf16` (passed as float *; element i of row
// m at index m * N + i of the element type).
inline float *y_offset(float *y, int64_t elems, bool ybf16) {
    return ybf16 ? reinterpret_cast<float *>(reinterpret_cast<uint16_t *>(y) + elems) : y + elems;
}

// Rows of x the decode kernels take (q4_0_gemv), and the largest M that
// q4_0_matmul sends to them rather than to the GEMM.
constexpr int64_t kGemvMaxM = 64;
constexpr int64_t kDecodeMaxM = 64;

// Decode GEMV for M <= kGemvMaxM (x, y point at row 0; row strides K and N).
// `workspace` (256-byte aligned, gemv_workspace_bytes(M, K) bytes) is used
// by the tensor-core decode only: 3 <= M <= kGemvMaxM, or M <= 2 with
// K > 65536.
// gemv_shape_supported: the launch grids of the path the shape takes stay
// within the device limits.
size_t gemv_workspace_bytes(int64_t M, int64_t K);
bool gemv_shape_supported(int64_t M, int64_t N, int64_t K);

// Grouped decode: independent problems y_g = x_g W_g^T with one row of x
// each, in as few launches as shared memory allows (all of x in the CTA, one
// weight stream).  grouped_decode_eligible: the problem can join a group
// (M == 1, K % 1024 == 0, K <= 65536, its plan fits).  The arrays hold G eligible
// problems; y_g has row stride N_g.
bool grouped_decode_eligible(int64_t M, int64_t N, int64_t K);
int grouped_decode_launches(int G, int64_t M, const int64_t *N, const int64_t *K);
cudaError_t launch_gemv_grouped(int G, const uint16_t *const *x, const uint8_t *const *wq, float *const *y,
                                bool ybf16, int64_t M, const int64_t *N, const int64_t *K, cudaStream_t s,
                                unsigned int *err);
cudaError_t launch_gemv(const uint16_t *x, const uint8_t *wq, float *y, bool ybf16, int64_t M, int64_t N,
                        int64_t K, void *workspace, cudaStream_t s, unsigned int *err);

// Tensor-core decode for M <= 64: x rounded once into binary16 MMA tiles in
// the workspace (gemv_tc_workspace_bytes(M, K) bytes, which also holds the
// split-K partial tiles and counters).  N <= 65535 * 128.
size_t gemv_tc_workspace_bytes(int64_t M, int64_t K);
cudaError_t launch_gemv_tc(const uint16_t *x, const uint8_t *wq, float *y, bool ybf16, int64_t M, int64_t N,
                           int64_t K, void *xtiles, cudaStream_t s, unsigned int *err);

// K % 32 == 0 but K % 256 != 0: W and x copied, zero-padded to K rounded up
// to 256 (padded_k), into the front of `workspace` (pad_bytes(M, N, K)
// bytes, 256-byte aligned); *xp and *wqp point at the copies.  Plain stream
// order (see pad.cu).
int64_t padded_k(int64_t K);
size_t pad_bytes(int64_t M, int64_t N, int64_t K);
cudaError_t launch_pad(const uint16_t *x, const uint8_t *wq, int64_t M, int64_t N, int64_t K, void *workspace,
                       uint16_t **xp, uint8_t **wqp, cudaStream_t s);

// tcgen05 GEMM.  `workspace` holds x rounded to binary16 and, when K is
// split (splits > 1), the fp32 partial tiles: gemm_workspace_bytes(M, N, K,
// splits) bytes.  gemm_splits picks the split for a device with `sms` SMs.
int gemm_splits(int64_t M, int64_t N, int64_t K, int sms);
// The launch plan of a GEMM with `splits` K splits on `sms` SMs: its x tile
// rows and whether the persistent form runs.
void gemm_plan(int64_t M, int64_t N, int64_t K, int sms, int splits, int *tile_rows, int *persistent);
bool gemm_shape_supported(int64_t M, int64_t N, int64_t K);
size_t gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, int splits);
cudaError_t launch_gemm(const uint16_t *x, const uint8_t *wq, float *y, bool ybf16, int64_t M, int64_t N,
                        int64_t K, void *workspace, int splits, cudaStream_t s, unsigned int *err);

}  // namespace q4_0
