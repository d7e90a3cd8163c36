// pad.cu -- K that is a multiple of 32 but not of 256.
//
// A Q4_0 row holds K / 32 blocks of 18 bytes.  The streaming kernels move
// rows and tiles with TMA and bulk copies, which need 16-byte-aligned row
// strides: K / 32 a multiple of 8, i.e. K % 256 == 0.  For any other K the
// dispatcher first copies W and x into a zero-padded layout with
// Kp = K rounded up to 256: the extra blocks are all zero (d = +0, codes 0,
// so every extra weight is 0) and the extra x elements are zero, which leaves
// every dot product unchanged.  The padded matmul then runs on the regular
// kernels.  This costs one extra pass over W per call; it serves shapes
// outside the 256-multiples, not the hot configurations.
//
// Ordering: the streaming kernels read weights before their dependency wait
// (no kernel of this library writes weights a dependent matmul may read).
// The padding kernels do write weights, so they are launched without
// programmatic dependent launch and trigger nothing early: the first starts
// after everything before it on the stream has finished, the second after
// the first, and a matmul kernel launched next cannot start before the second
// has exited, by which time the padded weights are complete.
#include <cuda_runtime.h>

#include "q4_0_internal.h"
#include "q4_0_ptx.cuh"

namespace q4_0 {
namespace {

// rows of `in_h` halfwords -> rows of `out_h` halfwords, zero-filled (Q4_0
// rows are 18-byte blocks, so halfwords are their natural unit of alignment)
__global__ void __launch_bounds__(256) pad_rows_kernel(const uint16_t *__restrict__ in, uint16_t *__restrict__ out,
                                                       int64_t rows, int64_t in_h, int64_t out_h) {
    const int64_t total = rows * out_h;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / out_h, j = i - r * out_h;
        out[i] = j < in_h ? in[r * in_h + j] : (uint16_t)0;
    }
}

cudaError_t pad_rows(const uint16_t *in, uint16_t *out, int64_t rows, int64_t in_h, int64_t out_h, int sms,
                     cudaStream_t s) {
    const int64_t total = rows * out_h;
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = (int64_t)(sms > 0 ? sms : 1) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    pad_rows_kernel<<<(unsigned)blocks, 256, 0, s>>>(in, out, rows, in_h, out_h);  // plain stream order
    return cudaGetLastError();
}

}  // namespace

int64_t padded_k(int64_t K) { return (K + 255) / 256 * 256; }

size_t pad_bytes(int64_t M, int64_t N, int64_t K) {
    if (K % 256 == 0) return 0;
    const int64_t kp = padded_k(K);
    const size_t w = (size_t)N * (size_t)(kp / 32) * 18;
    const size_t x = (size_t)M * (size_t)kp * 2;
    return (w + 255) / 256 * 256 + (x + 255) / 256 * 256;
}

cudaError_t launch_pad(const uint16_t *x, const uint8_t *wq, int64_t M, int64_t N, int64_t K, void *workspace,
                       uint16_t **xp, uint8_t **wqp, cudaStream_t s) {
    const int64_t kp = padded_k(K);
    const size_t wbytes = ((size_t)N * (size_t)(kp / 32) * 18 + 255) / 256 * 256;
    *wqp = static_cast<uint8_t *>(workspace);
    *xp = reinterpret_cast<uint16_t *>(static_cast<uint8_t *>(workspace) + wbytes);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int sms = device_sm_count(dev);
    e = pad_rows(reinterpret_cast<const uint16_t *>(wq), reinterpret_cast<uint16_t *>(*wqp), N, (K / 32) * 9,
                 (kp / 32) * 9, sms, s);
    if (e != cudaSuccess) return e;
    return pad_rows(x, *xp, M, K, kp, sms, s);
}

}  // namespace q4_0
