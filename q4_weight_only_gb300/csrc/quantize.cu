// quantize.cu -- fp32 weights -> Q4_0 blocks on the device.
//
// "Vertical disaggregation: maximizing model throughput on heterogeneous
// silicon", section "Every cycle counts: custom kernels": CPU and GPU share
// one Q4_0 weight format.  This kernel writes that format: per block of 32
// weights, d = (signed max-|w| element, first index on ties) / -8 in fp32,
// stored as binary16 (round to nearest even); q = clamp(round(w / d) + 8, 0,
// 15) with the fp32 d, IEEE division and round-half-away-from-zero; byte
// 2 + j holds q[j] in its low nibble and q[j + 16] in its high nibble.
// Off the hot path (once per weight load); one thread per block.
//
// This translation unit must not be built with fast-math: the codes depend
// on correctly rounded division and on roundf's tie rule.
#include <cuda_fp16.h>

#include "q4_0_internal.h"

namespace q4_0 {

__global__ void __launch_bounds__(256) quantize_kernel(const float *__restrict__ w,
                                                       uint8_t *__restrict__ wq,
                                                       int64_t nblocks) {
    const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (g >= nblocks) return;
    const float4 *src = reinterpret_cast<const float4 *>(w + g * 32);
    float v[32];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float4 t = __ldg(src + i);
        v[4 * i + 0] = t.x;
        v[4 * i + 1] = t.y;
        v[4 * i + 2] = t.z;
        v[4 * i + 3] = t.w;
    }
    float amax = fabsf(v[0]), wmax = v[0];
#pragma unroll
    for (int j = 1; j < 32; ++j) {
        if (fabsf(v[j]) > amax) {  // strict: the first index keeps a tie
            amax = fabsf(v[j]);
            wmax = v[j];
        }
    }
    uint16_t dbits = 0;
    uint32_t q[32];
    if (amax == 0.0f) {
#pragma unroll
        for (int j = 0; j < 32; ++j) q[j] = 8;
    } else {
        const float d = __fdiv_rn(wmax, -8.0f);
        dbits = __half_as_ushort(__float2half_rn(d));
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            int c = (int)roundf(__fdiv_rn(v[j], d)) + 8;
            c = c < 0 ? 0 : (c > 15 ? 15 : c);
            q[j] = (uint32_t)c;
        }
    }
    uint16_t *dst = reinterpret_cast<uint16_t *>(wq + g * 18);
    dst[0] = dbits;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t lo = q[2 * i] | (q[2 * i + 16] << 4);
        const uint32_t hi = q[2 * i + 1] | (q[2 * i + 17] << 4);
        dst[1 + i] = (uint16_t)(lo | (hi << 8));
    }
}

cudaError_t launch_quantize(const float *w, uint8_t *wq, int64_t N, int64_t K, cudaStream_t s,
                            unsigned int * /*err*/) {
    const int64_t nblocks = N * (K / 32);
    const int threads = 256;
    const int64_t grid = (nblocks + threads - 1) / threads;
    if (grid > 0x7FFFFFFF) return cudaErrorInvalidValue;
    quantize_kernel<<<(unsigned)grid, threads, 0, s>>>(w, wq, nblocks);
    return cudaGetLastError();
}

}  // namespace q4_0
