// gemv.cu -- decode GEMV y[m][n] = sum_k w[n][k] x[m][k] for small M.
//
// "Vertical disaggregation: maximizing model throughput on heterogeneous
// silicon", section "Every cycle counts: custom kernels": the Q4_0 kernels
// are built from nibble unpack, dot product, scale apply and batch decode,
// over the weight format the CPU shares.  Decode is bound by streaming the
// 0.5625 bytes per weight once from HBM; this kernel is written for that:
//
//   * one CTA per SM owns a contiguous range of weight rows (the rows are
//     contiguous in memory, so the CTA streams one contiguous byte range);
//   * work items are (pair of rows, chunk of 1024 weights); each warp owns
//     every 16th item and streams it with 1-D bulk TMA copies into its own
//     4-slot shared-memory ring (no CTA-wide synchronisation in the loop);
//   * lane (r, p) of a warp handles block pair p of row r of the item: nine
//     conflict-free 32-bit shared loads, nibble unpack into fp16 pairs with
//     the 0x6400 exponent trick, q - 8 exactly in fp16, and packed fp16
//     FMAs against x (pre-scaled per block by a power of two so that the
//     fp16 partial sums of one block cannot overflow);
//   * scale apply per block in fp32: acc += partial * d * 2^e;
//   * per item, a fixed butterfly over 16 lanes; per row, a fixed-order sum
//     over chunks -- the result does not depend on timing.
//
// x (M rows, all of K) is converted into shared memory once per CTA, so the
// kernel reads nothing but the weights, x and writes y.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "q4_0_internal.h"
#include "q4_0_ptx.cuh"

namespace q4_0 {
namespace {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kSlots = 4;                          // ring depth per warp
constexpr int kChunkPairs = 16;                    // block pairs per item row (1024 weights)
constexpr int kPairBytes = 36;                     // two Q4_0 blocks
constexpr int kRowChunkBytes = kChunkPairs * kPairBytes;  // 576
constexpr int kSlotBytes = 2 * kRowChunkBytes;            // two rows: 1152

struct GemvArgs {
    int64_t N, K;
    int P;         // block pairs per row (K / 64)
    int C;         // chunks per row
    int nb;        // blocks per row (K / 32)
    int mrows;     // valid x rows in this launch
    uint32_t off_sx, off_ring, off_bars, off_part, off_flag;
};

__device__ __forceinline__ half2 u2h(uint32_t u) {
    return *reinterpret_cast<half2 *>(&u);
}
__device__ __forceinline__ uint32_t h2u(half2 h) {
    return *reinterpret_cast<uint32_t *>(&h);
}

// One Q4_0 block (scale bits + four code words) against MT rows of x.
template <int MT>
__device__ __forceinline__ void block_dot(uint32_t dbits, const uint32_t (&Q)[4],
                                          const uint4 *__restrict__ xq, int P,
                                          const float *__restrict__ sxb, int nb,
                                          float (&acc)[MT]) {
    const uint32_t kMagic = 0x64006400u;  // two fp16 1024.0
    const half2 k1032 = __floats2half2_rn(1032.0f, 1032.0f);
    const half2 k1152 = __floats2half2_rn(1152.0f, 1152.0f);
    half2 v[16];
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
        const uint32_t q = Q[wi];
        const uint32_t q8 = q >> 8;
        // lanes hold (element 4wi, 4wi+2), (16(4wi+16), 16(4wi+18)), (4wi+1, 4wi+3), (16(4wi+17), 16(4wi+19))
        v[4 * wi + 0] = __hsub2(u2h((q & 0x000F000Fu) | kMagic), k1032);
        v[4 * wi + 1] = __hsub2(u2h((q & 0x00F000F0u) | kMagic), k1152);
        v[4 * wi + 2] = __hsub2(u2h((q8 & 0x000F000Fu) | kMagic), k1032);
        v[4 * wi + 3] = __hsub2(u2h((q8 & 0x00F000F0u) | kMagic), k1152);
    }
    const float d = __half2float(__ushort_as_half((unsigned short)dbits));
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        const uint4 *xp = xq + (size_t)m * 8 * P;
        half2 a0 = __floats2half2_rn(0.f, 0.f), a1 = a0;
#pragma unroll
        for (int wi = 0; wi < 4; ++wi) {
            const uint4 X = xp[wi * P];
            a0 = __hfma2(v[4 * wi + 0], u2h(X.x), a0);
            a1 = __hfma2(v[4 * wi + 1], u2h(X.y), a1);
            a0 = __hfma2(v[4 * wi + 2], u2h(X.z), a0);
            a1 = __hfma2(v[4 * wi + 3], u2h(X.w), a1);
        }
        const float2 f0 = __half22float2(a0), f1 = __half22float2(a1);
        const float s = (f0.x + f0.y) + (f1.x + f1.y);
        acc[m] = fmaf(s, d * sxb[(size_t)m * nb], acc[m]);
    }
}

template <int MT>
__global__ void __launch_bounds__(kThreads, 1)
    gemv_kernel(const uint16_t *__restrict__ x, const uint8_t *__restrict__ wq,
                float *__restrict__ y, const GemvArgs a, unsigned int *err) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint4 *xs = reinterpret_cast<uint4 *>(smem);  // [MT][8][P] quads of half2
    float *sx = reinterpret_cast<float *>(smem + a.off_sx);  // [MT][nb] 2^e
    uint8_t *ring = smem + a.off_ring;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + a.off_bars);
    float *part = reinterpret_cast<float *>(smem + a.off_part);  // [rows][C][MT]
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + a.off_flag);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int P = a.P, C = a.C, nb = a.nb;
    const int64_t r0 = (int64_t)blockIdx.x * a.N / gridDim.x;
    const int64_t r1 = (int64_t)(blockIdx.x + 1) * a.N / gridDim.x;
    const int nrows = (int)(r1 - r0);
    const int items = ((nrows + 1) >> 1) * C;
    const int64_t rowbytes = (int64_t)nb * 18;

    if (tid < kWarps * kSlots) mbar_init(&bars[tid], 1);
    if (tid == 0) *abort_flag = 0;
    mbar_fence_init();
    __syncthreads();

    const int my_items = items > warp ? (items - warp + kWarps - 1) / kWarps : 0;
    uint8_t *my_ring = ring + warp * kSlots * kSlotBytes;
    uint64_t *my_bars = bars + warp * kSlots;

    auto issue = [&](int j) {
        const int it = warp + kWarps * j;
        const int pr = it / C, c = it - pr * C;
        const int64_t rowA = r0 + 2 * pr;
        const int pairs = min(kChunkPairs, P - c * kChunkPairs);
        const uint32_t bytes = (uint32_t)pairs * kPairBytes;
        const bool hasB = rowA + 1 < r1;
        uint8_t *dst = my_ring + (j % kSlots) * kSlotBytes;
        uint64_t *bar = my_bars + (j % kSlots);
        const uint8_t *src = wq + rowA * rowbytes + (int64_t)c * kRowChunkBytes;
        mbar_arrive_expect_tx(bar, hasB ? 2 * bytes : bytes);
        bulk_g2s(dst, src, bytes, bar);
        if (hasB) bulk_g2s(dst + kRowChunkBytes, src + rowbytes, bytes, bar);
    };
    if (lane == 0) {
        for (int j = 0; j < kSlots && j < my_items; ++j) issue(j);
    }

    // x -> shared memory, per (row m, block b): e = exponent of max|x| so
    // that |x * 2^-e| < 1; quads of half2 in the order block_dot reads them;
    // the high-nibble lanes carry an extra 1/16 (their codes arrive as 16q).
    for (int t = tid; t < MT * nb; t += kThreads) {
        const int m = t / nb, b = t - m * nb;
        float xv[32];
        float amax = 0.f;
        if (m < a.mrows) {
            const uint4 *src = reinterpret_cast<const uint4 *>(x + (int64_t)m * a.K + (int64_t)b * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint4 u = __ldg(src + i);
                const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    xv[8 * i + 2 * h] = __uint_as_float(w4[h] << 16);
                    xv[8 * i + 2 * h + 1] = __uint_as_float(w4[h] & 0xFFFF0000u);
                }
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(xv[j]));
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) xv[j] = 0.f;
        }
        int e = 0;
        if (amax > 0.f) {
            frexpf(amax, &e);
            e = max(-125, min(127, e));
        }
        const float inv = ldexpf(1.0f, -e), inv16 = ldexpf(1.0f, -e - 4);
        sx[m * nb + b] = amax > 0.f ? ldexpf(1.0f, e) : 0.f;
        const int p = b >> 1, blk = b & 1;
#pragma unroll
        for (int wi = 0; wi < 4; ++wi) {
            uint4 o;
            o.x = h2u(__floats2half2_rn(xv[4 * wi] * inv, xv[4 * wi + 2] * inv));
            o.y = h2u(__floats2half2_rn(xv[4 * wi + 16] * inv16, xv[4 * wi + 18] * inv16));
            o.z = h2u(__floats2half2_rn(xv[4 * wi + 1] * inv, xv[4 * wi + 3] * inv));
            o.w = h2u(__floats2half2_rn(xv[4 * wi + 17] * inv16, xv[4 * wi + 19] * inv16));
            xs[(size_t)(m * 8 + blk * 4 + wi) * P + p] = o;
        }
    }
    __syncthreads();

    const int rr = lane >> 4, pp = lane & 15;
    int done = 0;
    for (int j = 0; j < my_items; ++j, ++done) {
        const int it = warp + kWarps * j;
        const int pr = it / C, c = it - pr * C;
        const int slot = j % kSlots;
        const bool ok = mbar_wait(my_bars + slot, (j / kSlots) & 1, abort_flag, err);
        if (!__all_sync(0xffffffffu, ok)) break;
        const int64_t n = r0 + 2 * pr + rr;
        const int p = c * kChunkPairs + pp;
        float acc[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[m] = 0.f;
        if (n < r1 && p < P) {
            const uint32_t *src = reinterpret_cast<const uint32_t *>(
                my_ring + slot * kSlotBytes + rr * kRowChunkBytes + pp * kPairBytes);
            uint32_t wv[9];
#pragma unroll
            for (int i = 0; i < 9; ++i) wv[i] = src[i];
            const uint32_t Q0[4] = {__funnelshift_r(wv[0], wv[1], 16), __funnelshift_r(wv[1], wv[2], 16),
                                    __funnelshift_r(wv[2], wv[3], 16), __funnelshift_r(wv[3], wv[4], 16)};
            const uint32_t Q1[4] = {wv[5], wv[6], wv[7], wv[8]};
            block_dot<MT>(wv[0] & 0xFFFFu, Q0, xs + p, P, sx + 2 * p, nb, acc);
            block_dot<MT>(wv[4] >> 16, Q1, xs + 4 * P + p, P, sx + 2 * p + 1, nb, acc);
        }
        __syncwarp();
        if (lane == 0 && j + kSlots < my_items) issue(j + kSlots);
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            float v = acc[m];
            v += __shfl_xor_sync(0xffffffffu, v, 8);
            v += __shfl_xor_sync(0xffffffffu, v, 4);
            v += __shfl_xor_sync(0xffffffffu, v, 2);
            v += __shfl_xor_sync(0xffffffffu, v, 1);
            acc[m] = v;
        }
        if (pp == 0 && n < r1) {
#pragma unroll
            for (int m = 0; m < MT; ++m) part[((2 * pr + rr) * C + c) * MT + m] = acc[m];
        }
    }
    if (done < my_items && lane == 0) {
        // abandoned: let the copies already issued land before exiting
        for (int j = done; j < my_items && j < done + kSlots; ++j)
            mbar_drain(my_bars + (j % kSlots), (j / kSlots) & 1);
    }
    __syncthreads();

    // fixed-order sum over chunks; consecutive threads write consecutive n
    for (int t = tid; t < nrows * a.mrows; t += kThreads) {
        const int m = t / nrows, r = t - m * nrows;
        float s = 0.f;
        for (int c = 0; c < C; ++c) s += part[(r * C + c) * MT + m];
        y[(int64_t)m * a.N + r0 + r] = s;
    }
}

struct GemvPlan {
    int mt;
    size_t smem;
    GemvArgs args;
};

GemvPlan plan_gemv(int mt, int64_t N, int64_t K, int grid) {
    GemvPlan p{};
    p.mt = mt;
    GemvArgs &a = p.args;
    a.N = N;
    a.K = K;
    a.P = (int)(K / 64);
    a.C = (a.P + kChunkPairs - 1) / kChunkPairs;
    a.nb = (int)(K / 32);
    const int64_t rows_cap = (N + grid - 1) / grid + 1;
    size_t off = (size_t)mt * 8 * a.P * 16;  // xs
    a.off_sx = (uint32_t)off;
    off += (size_t)mt * a.nb * 4;
    off = (off + 127) & ~(size_t)127;
    a.off_ring = (uint32_t)off;
    off += (size_t)kWarps * kSlots * kSlotBytes;
    a.off_bars = (uint32_t)off;
    off += (size_t)kWarps * kSlots * 8;
    a.off_part = (uint32_t)off;
    off += (size_t)rows_cap * a.C * mt * 4;
    off = (off + 15) & ~(size_t)15;
    a.off_flag = (uint32_t)off;
    off += 16;
    p.smem = off;
    return p;
}

template <int MT>
cudaError_t launch_mt(const uint16_t *x, const uint8_t *wq, float *y, const GemvPlan &p,
                      int grid, cudaStream_t s, unsigned int *err) {
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(gemv_kernel<MT>), (int)p.smem);
    if (e != cudaSuccess) return e;
    gemv_kernel<MT><<<grid, kThreads, p.smem, s>>>(x, wq, y, p.args, err);
    return cudaGetLastError();
}

constexpr size_t kSmemLimit = 227 * 1024;

}  // namespace

cudaError_t launch_gemv(const uint16_t *x, const uint8_t *wq, float *y, int64_t M, int64_t N,
                        int64_t K, cudaStream_t s, unsigned int *err) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int sms = device_sm_count(dev);
    if (sms <= 0) return cudaErrorInvalidDevice;
    const int64_t grid64 = (N + 1) / 2 < sms ? (N + 1) / 2 : sms;
    const int grid = (int)grid64;
    // rows of x per launch: the largest power of two <= 8 that covers M (or
    // fits shared memory); each launch streams the weights once
    int mt = 1;
    while (mt < 8 && mt < M) mt *= 2;
    while (mt > 1 && plan_gemv(mt, N, K, grid).smem > kSmemLimit) mt /= 2;
    if (plan_gemv(mt, N, K, grid).smem > kSmemLimit) return cudaErrorInvalidValue;
    for (int64_t m0 = 0; m0 < M; m0 += mt) {
        GemvPlan p = plan_gemv(mt, N, K, grid);
        p.args.mrows = (int)((M - m0) < mt ? (M - m0) : mt);
        const uint16_t *xm = x + m0 * K;
        float *ym = y + m0 * N;
        switch (mt) {
            case 1: e = launch_mt<1>(xm, wq, ym, p, grid, s, err); break;
            case 2: e = launch_mt<2>(xm, wq, ym, p, grid, s, err); break;
            case 4: e = launch_mt<4>(xm, wq, ym, p, grid, s, err); break;
            default: e = launch_mt<8>(xm, wq, ym, p, grid, s, err); break;
        }
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace q4_0
