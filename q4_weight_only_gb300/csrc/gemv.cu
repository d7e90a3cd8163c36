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
//     the 0x6400 exponent trick (q - 8 exactly), widened to fp32 and
//     multiplied in fp32 with x held as binary16 (pre-scaled per block by a
//     power of two so that the block's maximum sits just below 1);
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
    int64_t ldy;   // row stride of y (the full N when N is covered by several launches)
    int P;         // block pairs per row (K / 64)
    int C;         // chunks per row
    int nb;        // blocks per row (K / 32)
    int mrows;     // valid x rows in this launch
    int ybf16;     // y is bfloat16 (else fp32)
    uint32_t off_sx, off_ring, off_bars, off_part, off_flag;
};

__device__ __forceinline__ half2 u2h(uint32_t u) {
    return *reinterpret_cast<half2 *>(&u);
}
__device__ __forceinline__ uint32_t h2u(half2 h) {
    return *reinterpret_cast<uint32_t *>(&h);
}

// One Q4_0 block (scale bits + four code words) against MT rows of x.  The
// codes become exact binary16 integers (q - 8 for the low nibbles, 16 (q - 8)
// for the high ones, which need no shift), are widened to fp32 and
// multiplied by the binary16 x values in fp32; the high-nibble sums take the
// exact factor 1/16 at the end.  Scale apply: one fp32 FMA per block.
template <int MT>
__device__ __forceinline__ void block_dot(uint32_t dbits, const uint32_t (&Q)[4],
                                          const uint4 *__restrict__ xq, int P,
                                          const float *__restrict__ sxb, int nb,
                                          float (&acc)[MT]) {
    const uint32_t kMagic = 0x64006400u;  // two fp16 1024.0
    const half2 k1032 = __floats2half2_rn(1032.0f, 1032.0f);
    const half2 k1152 = __floats2half2_rn(1152.0f, 1152.0f);
    float2 v[16];
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
        const uint32_t q = Q[wi];
        const uint32_t q8 = q >> 8;
        // pairs hold (element 4wi, 4wi+2), (16(4wi+16), 16(4wi+18)), (4wi+1, 4wi+3), (16(4wi+17), 16(4wi+19))
        v[4 * wi + 0] = __half22float2(__hsub2(u2h((q & 0x000F000Fu) | kMagic), k1032));
        v[4 * wi + 1] = __half22float2(__hsub2(u2h((q & 0x00F000F0u) | kMagic), k1152));
        v[4 * wi + 2] = __half22float2(__hsub2(u2h((q8 & 0x000F000Fu) | kMagic), k1032));
        v[4 * wi + 3] = __half22float2(__hsub2(u2h((q8 & 0x00F000F0u) | kMagic), k1152));
    }
    const float d = __half2float(__ushort_as_half((unsigned short)dbits));
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        const uint4 *xp = xq + (size_t)m * 8 * P;
        float lo0 = 0.f, lo1 = 0.f, hi0 = 0.f, hi1 = 0.f;
#pragma unroll
        for (int wi = 0; wi < 4; ++wi) {
            const uint4 X = xp[wi * P];
            const float2 x0 = __half22float2(u2h(X.x)), x1 = __half22float2(u2h(X.y));
            const float2 x2 = __half22float2(u2h(X.z)), x3 = __half22float2(u2h(X.w));
            lo0 = fmaf(v[4 * wi + 0].x, x0.x, lo0);
            lo1 = fmaf(v[4 * wi + 0].y, x0.y, lo1);
            hi0 = fmaf(v[4 * wi + 1].x, x1.x, hi0);
            hi1 = fmaf(v[4 * wi + 1].y, x1.y, hi1);
            lo0 = fmaf(v[4 * wi + 2].x, x2.x, lo0);
            lo1 = fmaf(v[4 * wi + 2].y, x2.y, lo1);
            hi0 = fmaf(v[4 * wi + 3].x, x3.x, hi0);
            hi1 = fmaf(v[4 * wi + 3].y, x3.y, hi1);
        }
        const float s = (lo0 + lo1) + 0.0625f * (hi0 + hi1);
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

    const uint64_t policy = l2_evict_first_policy();  // weights are read once
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
        bulk_g2s_hint(dst, src, bytes, bar, policy);
        if (hasB) bulk_g2s_hint(dst + kRowChunkBytes, src + rowbytes, bytes, bar, policy);
    };
    pdl_launch_dependents();
    if (lane == 0) {
        for (int j = 0; j < kSlots && j < my_items; ++j) issue(j);
    }
    pdl_wait();

    // x -> shared memory, per (row m, block b): e = exponent of max|x| so
    // that |x * 2^-e| < 1 (binary16: exact down to 2^-14 of the block's
    // maximum, absolute error <= 2^(e-25) below); quads of half2 in the order
    // block_dot reads them.
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
        const float inv = ldexpf(1.0f, -e);
        sx[m * nb + b] = amax > 0.f ? ldexpf(1.0f, e) : 0.f;
        const int p = b >> 1, blk = b & 1;
#pragma unroll
        for (int wi = 0; wi < 4; ++wi) {
            uint4 o;
            o.x = h2u(__floats2half2_rn(xv[4 * wi] * inv, xv[4 * wi + 2] * inv));
            o.y = h2u(__floats2half2_rn(xv[4 * wi + 16] * inv, xv[4 * wi + 18] * inv));
            o.z = h2u(__floats2half2_rn(xv[4 * wi + 1] * inv, xv[4 * wi + 3] * inv));
            o.w = h2u(__floats2half2_rn(xv[4 * wi + 17] * inv, xv[4 * wi + 19] * inv));
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
        store_y(y, (int64_t)m * a.ldy + r0 + r, s, a.ybf16 != 0);
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
    a.ldy = N;
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
    return launch_pdl(gemv_kernel<MT>, dim3(grid), dim3(kThreads), p.smem, s, x, wq, y, p.args, err);
}

constexpr size_t kSmemLimit = 227 * 1024;

// ---------------------------------------------------------------------------
// Integer-dot decode kernel (M <= 2, K % 1024 == 0).
//
// x is turned, per 32-element block, into 15-bit fixed point X = round(x *
// 2^(14-e)) with 2^e > max|x| of the block, split into a signed high byte and
// an unsigned low byte (X = 256 Xh + Xl).  A Q4_0 block then needs
//   sum_j (q_j - 8) x_j = 2^(e-14) * (256 * sum q Xh + sum q Xl - 8 sum X),
// two exact 4-way byte dot products (dp4a) per four weights, the -8 sum X
// term precomputed once per block of x.  Scale apply: one fp32 FMA per block
// with d * 2^(e-14).  The integer sums are exact (|.| < 2^24), so the only
// rounding beyond fp32 accumulation is X's fixed point for elements far below
// their block's maximum.
//
// Thread (rs, tc) owns G block pairs (64 weights each) of every c-th row:
// their x bytes stay in registers for the whole kernel.  A producer warp
// streams stages of R whole rows (contiguous bytes) with one bulk TMA copy
// each; a row's pair partials are reduced by 16/G-lane butterflies into P/16
// partials, summed in order at the end.
// ---------------------------------------------------------------------------
namespace dp {

// One CTA per SM holding x in registers.  With one row of x a thread owns
// G = 2 block pairs of a row (the per-stage overhead -- wait, release,
// reduction, partial store -- is paid once per 128 weights); with two rows
// the x registers of one pair per thread are what the register file allows.
template <int MT>
struct Limits {
    static constexpr int kG = MT == 1 ? 2 : 1;       // block pairs per thread
    static constexpr int kRed = 16 / kG;              // lanes per partial (P / 16 partials per row)
    static constexpr int kThreads = MT == 1 ? 448 : 640;
    static constexpr int kCtasPerSm = 1;
    static constexpr size_t kSmem = 227 * 1024;
};

struct Args {
    int64_t N, K;
    int64_t ldy;  // row stride of y
    int P, c, T, R, S, rowbytes, H, mrows, ybf16;
    uint32_t stage_bytes, off_x, off_bars, off_part;
};

// Fixed-point x of one block pair, as kept in shared memory and registers:
// words 0-15 Xh bytes (block 0 words 0-7, block 1 words 8-15), 16-31 Xl
// bytes, 32-33 -8 * sum X per block, 34-35 2^(e-14) per block.
constexpr int kPairWords = 36;

template <int MT>
struct XReg {
    uint32_t h[MT][16];
    uint32_t l[MT][16];
    int ncorr[MT][2];
    float xs[MT][2];
};

__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp4a_uu(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Sixteen elements (half `part` of block b of x row m) -> fixed point,
// written into the pair record; the two threads of a block (consecutive
// lanes) agree on the block's exponent and sum through a shuffle.  `live` is
// false for lanes past the end (they still take part in the shuffles).  The
// two 16-byte loads are issued by load_part, ahead of every conversion of the
// thread, so that a CTA pays one load round trip for all of x.
__device__ __forceinline__ void load_part(const uint16_t *__restrict__ xrow, int b, int part, bool live,
                                          uint4 (&u)[2]) {
    if (live && xrow) {
        const uint4 *src = reinterpret_cast<const uint4 *>(xrow + (int64_t)b * 32) + 2 * part;
        u[0] = __ldg(src);
        u[1] = __ldg(src + 1);
    } else {
        u[0] = make_uint4(0u, 0u, 0u, 0u);
        u[1] = u[0];
    }
}

__device__ __forceinline__ void convert_part(const uint4 (&u)[2], int b, int part, bool live,
                                             uint32_t *__restrict__ rec) {
    float xv[16];
    const uint32_t w8[8] = {u[0].x, u[0].y, u[0].z, u[0].w, u[1].x, u[1].y, u[1].z, u[1].w};
#pragma unroll
    for (int h = 0; h < 8; ++h) {
        xv[2 * h] = __uint_as_float(w8[h] << 16);
        xv[2 * h + 1] = __uint_as_float(w8[h] & 0xFFFF0000u);
    }
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(xv[j]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    int e = 0;
    if (amax > 0.f) {
        frexpf(amax, &e);
        e = max(-100, min(127, e));
    }
    const float up = amax > 0.f ? ldexpf(1.0f, 14 - e) : 0.f;
    int X[16], sum = 0;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        X[j] = __float2int_rn(xv[j] * up);
        sum += X[j];
    }
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    if (!live) return;
    const int blk = b & 1;
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        const int wd = 4 * part + h;  // word: elements 4 wd .. 4 wd + 3
        const int *Xw = X + 4 * h;
        // bytes 1 (high) and 0 (low) of the four 16-bit fixed-point values
        rec[blk * 8 + wd] = __byte_perm(__byte_perm(Xw[0], Xw[1], 0x0051), __byte_perm(Xw[2], Xw[3], 0x0051), 0x5410);
        rec[16 + blk * 8 + wd] =
            __byte_perm(__byte_perm(Xw[0], Xw[1], 0x0040), __byte_perm(Xw[2], Xw[3], 0x0040), 0x5410);
    }
    if (part == 0) {
        reinterpret_cast<int *>(rec)[32 + blk] = -8 * sum;
        reinterpret_cast<float *>(rec)[34 + blk] = amax > 0.f ? ldexpf(1.0f, e - 14) : 0.f;
    }
}

// One Q4_0 block against MT rows of x: v[m] += d * 2^(e-14) * T.
template <int MT>
__device__ __forceinline__ void block_dp(uint32_t dbits, const uint32_t (&Q)[4], const XReg<MT> &r,
                                         int blk, float (&v)[MT]) {
    uint32_t lo[4], hi[4];
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
        lo[wi] = Q[wi] & 0x0F0F0F0Fu;         // elements 4wi .. 4wi+3
        hi[wi] = (Q[wi] >> 4) & 0x0F0F0F0Fu;  // elements 16+4wi .. 16+4wi+3
    }
    const float d = __half2float(__ushort_as_half((unsigned short)dbits));
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        int ah = 0, al = r.ncorr[m][blk];
#pragma unroll
        for (int wi = 0; wi < 4; ++wi) {
            ah = dp4a_us(lo[wi], r.h[m][blk * 8 + wi], ah);
            al = dp4a_uu(lo[wi], r.l[m][blk * 8 + wi], al);
            ah = dp4a_us(hi[wi], r.h[m][blk * 8 + 4 + wi], ah);
            al = dp4a_uu(hi[wi], r.l[m][blk * 8 + 4 + wi], al);
        }
        const int T = ah * 256 + al;
        v[m] = fmaf((float)T, d * r.xs[m][blk], v[m]);
    }
}

// ---- pieces shared by the one-problem and the grouped kernel ----

// x (MT rows of K = 64 P elements; rows >= mrows read as zero) -> the pair
// records at xsm, by the T compute threads.  Every thread issues the loads
// of up to kParts parts before converting any, so a CTA pays one load round
// trip for each kParts * T parts.  Trip counts are warp-uniform.
template <int MT>
__device__ __forceinline__ void convert_x(const uint16_t *__restrict__ x, int64_t K, int P, int mrows,
                                          uint32_t *__restrict__ xsm, int tid, int lane, int T) {
    static_assert(MT <= 2, "the row of a block is blk_id >= nb");
    constexpr int kParts = 4;
    const int nb = 2 * P;
    const int nparts = 2 * MT * nb;  // two threads per 32-element block
    for (int t0 = tid - lane; t0 < nparts; t0 += kParts * T) {
        uint4 u[kParts][2];
#pragma unroll
        for (int k = 0; k < kParts; ++k) {
            if (t0 + k * T < nparts) {
                const int t = t0 + k * T + lane;
                const int q = t < nparts ? t : nparts - 1;
                const int blk_id = q >> 1, m = blk_id >= nb ? 1 : 0;
                load_part(m < mrows ? x + (int64_t)m * K : nullptr, blk_id - m * nb, q & 1, t < nparts, u[k]);
            }
        }
#pragma unroll
        for (int k = 0; k < kParts; ++k) {
            if (t0 + k * T < nparts) {
                const int t = t0 + k * T + lane;
                const int q = t < nparts ? t : nparts - 1;
                const int blk_id = q >> 1, m = blk_id >= nb ? 1 : 0, b = blk_id - m * nb;
                convert_part(u[k], b, q & 1, t < nparts, xsm + ((size_t)m * P + (b >> 1)) * kPairWords);
            }
        }
    }
}

// The x registers of a thread that owns block pairs tc + g * tpr (g < G).
template <int MT>
__device__ __forceinline__ void load_xregs(const uint32_t *__restrict__ xsm, int P, int tpr, int tc,
                                           XReg<MT> (&xr)[Limits<MT>::kG]) {
#pragma unroll
    for (int g = 0; g < Limits<MT>::kG; ++g) {
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            const uint4 *rec = reinterpret_cast<const uint4 *>(xsm + ((size_t)m * P + tc + g * tpr) * kPairWords);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint4 u = rec[i], w = rec[4 + i];
                xr[g].h[m][4 * i] = u.x; xr[g].h[m][4 * i + 1] = u.y;
                xr[g].h[m][4 * i + 2] = u.z; xr[g].h[m][4 * i + 3] = u.w;
                xr[g].l[m][4 * i] = w.x; xr[g].l[m][4 * i + 1] = w.y;
                xr[g].l[m][4 * i + 2] = w.z; xr[g].l[m][4 * i + 3] = w.w;
            }
            const uint4 t = rec[8];
            xr[g].ncorr[m][0] = (int)t.x;
            xr[g].ncorr[m][1] = (int)t.y;
            xr[g].xs[m][0] = __uint_as_float(t.z);
            xr[g].xs[m][1] = __uint_as_float(t.w);
        }
    }
}

// The ring of weight stages as one thread consumes it.
struct Ring {
    const uint8_t *smem;  // slot 0
    uint64_t *full, *empty;
    volatile int *abort_flag;
    unsigned int *err;
    int S;                // slots
    uint32_t slot_bytes;  // bytes between slots
};

// nst stages of R whole rows (rowbytes each; the last stage last_rows rows):
// thread (rs, tc) copies its block pairs of row rs to registers, computes,
// then releases the stage to the producer -- only once the loaded words have
// been used, since the next bulk fill of the slot is an async-proxy write
// that must not overtake shared loads still in flight.  A row's pair sums
// are reduced over kRed lanes into H partials per row at part.  The loop is
// issue-bound at one pair per thread per stage, so the slot s, its phase ph
// (carried across calls) and the partials' address advance incrementally:
// a runtime division per stage cost about a tenth of the rate.  false when a
// wait gave up.
template <int MT>
__device__ __forceinline__ bool stream_rows(const Ring &r, int &s, uint32_t &ph, int nst, int last_rows, int R,
                                            int rowbytes, int H, int tpr, int tc, int rs, bool active, int lane,
                                            const XReg<MT> (&xr)[Limits<MT>::kG], float *__restrict__ part) {
    constexpr int G = Limits<MT>::kG, kRed = Limits<MT>::kRed;
    const uint8_t *my_row = r.smem + (size_t)rs * rowbytes + tc * 36;
    float *my_part = part + ((size_t)rs * H + tc / kRed) * MT;
    const int part_step = R * H * MT;
    for (int i = 0; i < nst; ++i) {
        const bool ok = mbar_wait(&r.full[s], ph, r.abort_flag, r.err);
        if (!__all_sync(0xffffffffu, ok)) return false;
        const int rows = i == nst - 1 ? last_rows : R;
        const bool valid = active && rs < rows;
        uint32_t wv[G][9];
        if (valid) {
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const uint32_t *src =
                    reinterpret_cast<const uint32_t *>(my_row + (uint32_t)s * r.slot_bytes + g * tpr * 36);
#pragma unroll
                for (int k = 0; k < 9; ++k) wv[g][k] = src[k];
            }
        }
        float v[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) v[m] = 0.f;
        if (valid) {
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const uint32_t *w = wv[g];
                const uint32_t Q0[4] = {__funnelshift_r(w[0], w[1], 16), __funnelshift_r(w[1], w[2], 16),
                                        __funnelshift_r(w[2], w[3], 16), __funnelshift_r(w[3], w[4], 16)};
                const uint32_t Q1[4] = {w[5], w[6], w[7], w[8]};
                block_dp<MT>(w[0] & 0xFFFFu, Q0, xr[g], 0, v);
                block_dp<MT>(w[4] >> 16, Q1, xr[g], 1, v);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&r.empty[s]);
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            float t = v[m];
#pragma unroll
            for (int o = kRed / 2; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
            v[m] = t;
        }
        if (valid && (lane & (kRed - 1)) == 0) {
#pragma unroll
            for (int m = 0; m < MT; ++m) my_part[m] = v[m];
        }
        my_part += part_step;
        if (++s == r.S) {
            s = 0;
            ph ^= 1;
        }
    }
    return true;
}

// Fixed-order sums over the H partials of each of a CTA's rows [r0, r1)
// (stages of R rows), stored to y (row stride ldy); consecutive threads
// write consecutive rows of a stage.
template <int MT>
__device__ __forceinline__ void row_sums(const float *__restrict__ part, int64_t r0, int64_t r1, int nst, int R,
                                         int H, int mrows, float *__restrict__ y, int64_t ldy, bool ybf16, int tid,
                                         int T) {
    const int local_rows = nst * R;
    for (int t = tid; t < local_rows * mrows; t += T) {
        const int m = t / local_rows, lr = t - m * local_rows;
        const int i = lr / R, rr = lr - i * R;
        const int64_t row = r0 + (int64_t)i * R;
        if (rr >= (int)(r1 - row < R ? r1 - row : R)) continue;
        float sum = 0.f;
        for (int h = 0; h < H; ++h) sum += part[((size_t)lr * H + h) * MT + m];
        store_y(y, (int64_t)m * ldy + row + rr, sum, ybf16);
    }
}

template <int MT>
__global__ void __launch_bounds__(Limits<MT>::kThreads, Limits<MT>::kCtasPerSm)
    gemv_dp4a_kernel(const uint16_t *__restrict__ x, const uint8_t *__restrict__ wq,
                     float *__restrict__ y, const Args a, unsigned int *err) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint32_t *xsm = reinterpret_cast<uint32_t *>(smem + a.off_x);  // [MT][P][36]
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + a.off_bars);
    uint64_t *empty = full + a.S;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + a.S);
    uint64_t *xready = empty + a.S + 1;  // x converted (the compute threads' signal to the producer)
    float *part = reinterpret_cast<float *>(smem + a.off_part);  // [rows][H][MT]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nwc = a.T >> 5;
    // CTA b owns the contiguous rows [r0, r1); stage i = rows r0 + i R ...
    const int64_t r0 = (int64_t)blockIdx.x * a.N / gridDim.x;
    const int64_t r1 = (int64_t)(blockIdx.x + 1) * a.N / gridDim.x;
    const int nst = (int)((r1 - r0 + a.R - 1) / a.R);
    auto stage_row0 = [&](int i) -> int64_t { return r0 + (int64_t)i * a.R; };
    auto stage_rows = [&](int i) -> int {
        const int64_t r = stage_row0(i);
        return (int)(r1 - r < a.R ? r1 - r : a.R);
    };
    // weights are streamed once: mark them first to leave L2 so that x and
    // y (small, reused by the next kernels) stay resident
    const uint64_t policy = l2_evict_first_policy();
    auto issue = [&](int i) {
        const int s = i % a.S;
        const uint32_t bytes = (uint32_t)stage_rows(i) * (uint32_t)a.rowbytes;
        mbar_arrive_expect_tx(&full[s], bytes);
        bulk_g2s_hint(smem + (size_t)s * a.stage_bytes, wq + stage_row0(i) * a.rowbytes, bytes, &full[s],
                      policy);
    };

    if (warp == nwc && lane == 0) {
        for (int i = 0; i < a.S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], nwc);
        }
        mbar_init(xready, 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();
    // trigger the next kernel before anything slow: issuing a bulk copy of a
    // stage takes a fraction of a microsecond
    pdl_launch_dependents();

    if (warp == nwc) {
        // Weights are read before pdl_wait(): no kernel of this library
        // writes Q4_0 weights while a dependent matmul may be running.  The
        // first stages go out at once; the rest of the ring waits until x is
        // converted: a CTA that starts after the previous kernel has ended
        // would otherwise find its x loads queued behind a ring's worth of
        // weight bytes arriving at the same SM, and such a late CTA decides
        // when the kernel ends.  With one row of x the rest of the ring's
        // first fill is requested into L2 meanwhile (no shared-memory
        // destination, so the SM's incoming path stays free for x); it then
        // arrives from L2 once x is ready.  Prefetching deeper than the ring,
        // or with two rows of x, measured slower.
        if (lane == 0) {
            constexpr int kPreWait = 3;
            const int pre = min(kPreWait, min(a.S, nst));
            for (int i = 0; i < pre; ++i) issue(i);
            if (MT == 1)
                for (int i = pre; i < a.S && i < nst; ++i)
                    bulk_prefetch_l2(wq + stage_row0(i) * a.rowbytes, (uint32_t)stage_rows(i) * (uint32_t)a.rowbytes,
                                     policy);
            pdl_wait();
            mbar_wait(xready, 0, abort_flag, err);
            for (int i = pre; i < a.S && i < nst; ++i) issue(i);
            int issued = min(a.S, nst);
            for (int i = a.S; i < nst; ++i) {
                if (!mbar_wait(&empty[i % a.S], ((i / a.S) & 1) ^ 1, abort_flag, err)) break;
                issue(i);
                ++issued;
            }
            for (int i = max(0, issued - a.S); i < issued; ++i)
                mbar_drain(&full[i % a.S], (i / a.S) & 1);
        }
        return;
    }

    // x -> fixed point in shared memory, once per CTA (overlaps the first copies)
    pdl_wait();
    convert_x<MT>(x, a.K, a.P, a.mrows, xsm, tid, lane, a.T);
    named_bar_sync(1, a.T);
    if (tid == 0) mbar_arrive(xready);

    // thread (rs, tc) owns block pairs tc + g TPR (g < G) of row slot rs
    const int tpr = a.P / Limits<MT>::kG;
    const int tc = tid % tpr, rs = tid / tpr;
    XReg<MT> xr[Limits<MT>::kG];
    load_xregs<MT>(xsm, a.P, tpr, tc, xr);
    const Ring ring{smem, full, empty, abort_flag, err, a.S, a.stage_bytes};
    int s = 0;
    uint32_t ph = 0;
    stream_rows<MT>(ring, s, ph, nst, (int)(r1 - r0 - (int64_t)(nst - 1) * a.R), a.R, a.rowbytes, a.H, tpr, tc, rs,
                    rs < a.c, lane, xr, part);
    named_bar_sync(1, a.T);
    row_sums<MT>(part, r0, r1, nst, a.R, a.H, a.mrows, y, a.ldy, a.ybf16 != 0, tid, a.T);
}

struct Plan {
    Args a;
    size_t smem;
    int threads;
    bool ok;
};

// One CTA per SM: c row slots of P / G threads (P = K / 64 block pairs), a
// producer warp, and as many row stages of about 29 KB as shared memory holds.
Plan make_plan(int mt, int64_t N, int64_t K, int grid) {
    Plan p{};
    Args &a = p.a;
    a.N = N;
    a.ldy = N;
    a.K = K;
    a.P = (int)(K / 64);
    p.ok = (K % 1024 == 0);
    if (!p.ok) return p;
    const int max_threads = mt == 1 ? Limits<1>::kThreads : Limits<2>::kThreads;
    const size_t smem_limit = mt == 1 ? Limits<1>::kSmem : Limits<2>::kSmem;
    const int budget = max_threads - 32;
    const int tpr = a.P / (mt == 1 ? Limits<1>::kG : Limits<2>::kG);  // threads per row slot
    a.c = max(1, budget / tpr);  // P % 16 == 0: row slots start on reduction-group boundaries
    a.T = ((a.c * tpr + 31) / 32) * 32;
    p.threads = a.T + 32;
    if (p.threads > max_threads || a.P % 16 != 0) {
        p.ok = false;
        return p;
    }
    a.rowbytes = (int)(K / 32 * 18);
    a.R = a.c;  // a stage is one row per row slot
    a.H = a.P / 16;
    a.stage_bytes = (uint32_t)a.R * (uint32_t)a.rowbytes;
    const int64_t rows_cap = ((N + grid - 1) / grid + a.R) / a.R * a.R;
    const size_t fixed = (size_t)mt * a.P * kPairWords * 4 + (size_t)rows_cap * a.H * mt * 4 + 16 * 8 + 64;
    int S = 8;
    while (S > 2 && (size_t)S * a.stage_bytes + fixed > smem_limit) --S;
    a.S = S;
    size_t off = (size_t)a.S * a.stage_bytes;
    off = (off + 127) & ~(size_t)127;
    a.off_x = (uint32_t)off;
    off += (size_t)mt * a.P * kPairWords * 4;
    a.off_bars = (uint32_t)off;
    off += (size_t)2 * a.S * 8 + 16;  // full[S], empty[S], then the abort flag and the x-ready barrier
    a.off_part = (uint32_t)off;
    off += (size_t)rows_cap * a.H * mt * 4;
    p.smem = off;
    p.ok = p.smem <= smem_limit;
    return p;
}

// One launch over n weight rows (all M = MT rows of x); y has row stride ldy.
template <int MT>
cudaError_t launch(const uint16_t *x, const uint8_t *wq, float *y, bool ybf16, int64_t n, int64_t ldy,
                   int64_t K, int sms, cudaStream_t s, unsigned int *err) {
    const int grid = (int)(n < sms ? n : sms);
    Plan p = make_plan(MT, n, K, grid);
    if (!p.ok) return cudaErrorInvalidValue;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(gemv_dp4a_kernel<MT>), (int)p.smem);
    if (e != cudaSuccess) return e;
    p.a.ybf16 = ybf16 ? 1 : 0;
    p.a.mrows = MT;
    p.a.ldy = ldy;
    return launch_pdl(gemv_dp4a_kernel<MT>, dim3(grid), dim3(p.threads), p.smem, s, x, wq, y, p.a, err);
}

bool fits(int mt, int64_t n, int64_t K, int sms) { return make_plan(mt, n, K, (int)(n < sms ? n : sms)).ok; }

// ---------------------------------------------------------------------------
// Grouped decode: up to kMaxGroup independent problems y_g = x_g W_g^T (one
// row of x each, each K_g % 1024 == 0) in one launch.  Every CTA owns the same share
// of rows of each problem; one producer ring streams the problems' stages
// back to back, so a step of several matrices pays the per-launch front
// (dependency release, x conversion) and tail (row sums) once instead of
// once per matrix.  x of every problem is converted at the start; each
// thread reloads its x registers when the stream moves on to the next
// problem.  Per row the arithmetic and the summation order are those of
// gemv_dp4a_kernel, so results equal the one-problem calls bit for bit.
// ---------------------------------------------------------------------------
constexpr int kMaxGroup = 8;

struct GroupItem {
    const uint16_t *x;
    const uint8_t *wq;
    float *y;   // element type per GroupArgs::ybf16
    int64_t N;
    int P, c, R, H, rowbytes;
    uint32_t off_x, off_part;  // this problem's x records and row partials in shared memory
};

struct GroupArgs {
    int G, S, T, mrows, ybf16;
    uint32_t slot_bytes, off_bars;
    GroupItem it[kMaxGroup];
};

template <int MT>
__global__ void __launch_bounds__(Limits<MT>::kThreads, Limits<MT>::kCtasPerSm)
    gemv_dp4a_grouped_kernel(const __grid_constant__ GroupArgs a, unsigned int *err) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + a.off_bars);
    uint64_t *empty = full + a.S;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + a.S);
    uint64_t *xready = empty + a.S + 1;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nwc = a.T >> 5;
    // this CTA's rows [r0, r1) of problem g and their stage count
    auto rows_of = [&](int g, int64_t &r0, int64_t &r1) {
        r0 = (int64_t)blockIdx.x * a.it[g].N / gridDim.x;
        r1 = (int64_t)(blockIdx.x + 1) * a.it[g].N / gridDim.x;
    };
    auto stages_of = [&](int g) -> int {
        int64_t r0, r1;
        rows_of(g, r0, r1);
        return (int)((r1 - r0 + a.it[g].R - 1) / a.it[g].R);
    };

    if (warp == nwc && lane == 0) {
        for (int i = 0; i < a.S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], nwc);
        }
        mbar_init(xready, 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();
    pdl_launch_dependents();

    if (warp == nwc) {
        // the stages of all problems in order, as the compute threads take them
        if (lane == 0) {
            const uint64_t policy = l2_evict_first_policy();
            struct Cursor {
                int g, i, nst;
                int64_t r0, r1;
            };
            auto seek = [&](Cursor &c) {  // first stage at or after (g, i)
                while (c.g < a.G) {
                    if (c.i == 0) {
                        rows_of(c.g, c.r0, c.r1);
                        c.nst = stages_of(c.g);
                    }
                    if (c.i < c.nst) return;
                    ++c.g;
                    c.i = 0;
                }
            };
            auto next = [&](Cursor &c) {
                ++c.i;
                seek(c);
            };
            auto stage = [&](const Cursor &c, int64_t &row, uint32_t &bytes) {
                const GroupItem &p = a.it[c.g];
                row = c.r0 + (int64_t)c.i * p.R;
                bytes = (uint32_t)(c.r1 - row < p.R ? c.r1 - row : p.R) * (uint32_t)p.rowbytes;
            };
            int total = 0;
            for (int g = 0; g < a.G; ++g) total += stages_of(g);
            Cursor cur{0, 0, 0, 0, 0};
            seek(cur);
            int j = 0;  // stages issued
            auto issue = [&]() {
                int64_t row;
                uint32_t bytes;
                stage(cur, row, bytes);
                const int s = j % a.S;
                mbar_arrive_expect_tx(&full[s], bytes);
                bulk_g2s_hint(smem + (size_t)s * a.slot_bytes, a.it[cur.g].wq + row * a.it[cur.g].rowbytes, bytes,
                              &full[s], policy);
                ++j;
                next(cur);
            };
            // as in the one-problem kernel: the first stages before the
            // dependency wait, the rest of the first ring fill into L2
            constexpr int kPreWait = 3;
            const int pre = min(kPreWait, min(a.S, total));
            while (j < pre) issue();
            if (MT == 1) {
                Cursor c = cur;
                for (int k = j; k < a.S && k < total; ++k) {
                    int64_t row;
                    uint32_t bytes;
                    stage(c, row, bytes);
                    bulk_prefetch_l2(a.it[c.g].wq + row * a.it[c.g].rowbytes, bytes, policy);
                    next(c);
                }
            }
            pdl_wait();
            mbar_wait(xready, 0, abort_flag, err);
            while (j < a.S && j < total) issue();
            while (j < total) {
                if (!mbar_wait(&empty[j % a.S], ((j / a.S) & 1) ^ 1, abort_flag, err)) break;
                issue();
            }
            for (int i = max(0, j - a.S); i < j; ++i) mbar_drain(&full[i % a.S], (i / a.S) & 1);
        }
        return;
    }

    // x of every problem -> fixed point in its records
    pdl_wait();
    for (int g = 0; g < a.G; ++g)
        convert_x<MT>(a.it[g].x, (int64_t)a.it[g].P * 64, a.it[g].P, a.mrows,
                      reinterpret_cast<uint32_t *>(smem + a.it[g].off_x), tid, lane, a.T);
    named_bar_sync(1, a.T);
    if (tid == 0) mbar_arrive(xready);

    // the problems' stages in order through one ring; the slot and its phase
    // carry over from one problem to the next
    const Ring ring{smem, full, empty, abort_flag, err, a.S, a.slot_bytes};
    int s = 0;
    uint32_t ph = 0;
    for (int g = 0; g < a.G; ++g) {
        const GroupItem &p = a.it[g];
        int64_t r0, r1;
        rows_of(g, r0, r1);
        const int nst = (int)((r1 - r0 + p.R - 1) / p.R);
        if (nst == 0) continue;
        // thread (rs, tc) owns block pairs tc + gg TPR of row slot rs of this problem
        const int tpr = p.P / Limits<MT>::kG;
        const int tc = tid % tpr, rs = tid / tpr;
        XReg<MT> xr[Limits<MT>::kG];
        load_xregs<MT>(reinterpret_cast<const uint32_t *>(smem + p.off_x), p.P, tpr, tc, xr);
        if (!stream_rows<MT>(ring, s, ph, nst, (int)(r1 - r0 - (int64_t)(nst - 1) * p.R), p.R, p.rowbytes, p.H,
                             tpr, tc, rs, rs < p.c, lane, xr, reinterpret_cast<float *>(smem + p.off_part)))
            break;
    }
    named_bar_sync(1, a.T);
    for (int g = 0; g < a.G; ++g) {
        const GroupItem &p = a.it[g];
        int64_t r0, r1;
        rows_of(g, r0, r1);
        row_sums<MT>(reinterpret_cast<const float *>(smem + p.off_part), r0, r1, (int)((r1 - r0 + p.R - 1) / p.R),
                     p.R, p.H, a.mrows, p.y, p.N, a.ybf16 != 0, tid, a.T);
    }
}

// Shared-memory plan of a group: the ring (S slots of the largest stage),
// each problem's x records and row partials, the barriers.  false when the
// problems do not fit with at least kMinGroupStages stages (a shallower ring
// streams slower than splitting the group).
bool plan_group(int mt, int grid, int G, const int64_t *N, const int64_t *K, GroupArgs &a, size_t &smem,
                int &threads) {
    const int max_threads = mt == 1 ? Limits<1>::kThreads : Limits<2>::kThreads;
    const size_t smem_limit = mt == 1 ? Limits<1>::kSmem : Limits<2>::kSmem;
    const int gsz = mt == 1 ? Limits<1>::kG : Limits<2>::kG;
    const int budget = max_threads - 32;
    a.G = G;
    uint32_t slot = 0;
    int T = 0;
    size_t fixed = 0;
    for (int g = 0; g < G; ++g) {
        GroupItem &p = a.it[g];
        if (K[g] % 1024 != 0 || N[g] < 1) return false;
        p.N = N[g];
        p.P = (int)(K[g] / 64);
        const int tpr = p.P / gsz;
        p.c = max(1, budget / tpr);
        if (p.c * tpr > budget) return false;
        T = max(T, ((p.c * tpr + 31) / 32) * 32);
        p.R = p.c;
        p.H = p.P / 16;
        p.rowbytes = (int)(K[g] / 32 * 18);
        slot = max(slot, (uint32_t)(p.R * p.rowbytes));
        const int64_t rows_cap = ((N[g] + grid - 1) / grid + p.R) / p.R * p.R;
        fixed += (size_t)mt * p.P * kPairWords * 4 + (size_t)rows_cap * p.H * mt * 4;
    }
    slot = (slot + 127) & ~127u;
    constexpr int kMinGroupStages = 5;
    int S = 8;
    while (S > kMinGroupStages && (size_t)S * slot + fixed + 16 * 8 + 64 > smem_limit) --S;
    size_t off = (size_t)S * slot;
    for (int g = 0; g < G; ++g) {
        GroupItem &p = a.it[g];
        p.off_x = (uint32_t)off;
        off += (size_t)mt * p.P * kPairWords * 4;
    }
    for (int g = 0; g < G; ++g) {
        GroupItem &p = a.it[g];
        p.off_part = (uint32_t)off;
        const int64_t rows_cap = ((N[g] + grid - 1) / grid + p.R) / p.R * p.R;
        off += (size_t)rows_cap * p.H * mt * 4;
    }
    off = (off + 15) & ~(size_t)15;
    a.off_bars = (uint32_t)off;
    off += (size_t)2 * S * 8 + 16;
    a.S = S;
    a.T = T;
    a.slot_bytes = slot;
    smem = off;
    threads = T + 32;
    return smem <= smem_limit && threads <= max_threads;
}

template <int MT>
cudaError_t launch_group(const GroupArgs &a0, size_t smem, int threads, int grid, cudaStream_t s,
                         unsigned int *err) {
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(gemv_dp4a_grouped_kernel<MT>), (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(gemv_dp4a_grouped_kernel<MT>, dim3(grid), dim3(threads), smem, s, a0, err);
}

}  // namespace dp

}  // namespace

// The largest share of N (N halved until it fits) whose plan fits shared
// memory: the per-row partial sums a CTA keeps grow with the rows it owns, so
// a very tall matrix runs as several launches.  0 when none fits.
template <class Fits>
int64_t rows_per_launch(int64_t N, Fits fits) {
    for (int64_t n = N;; n = (n + 1) / 2) {
        if (fits(n)) return n;
        if (n == 1) return 0;
    }
}

// M <= 2 with K up to this runs on the CUDA cores (x of one row is held in
// shared memory); larger K goes to the tensor-core decode, which streams x.
constexpr int64_t kDecodeMaxK = 65536;

bool decode_on_tensor_cores(int64_t M, int64_t K) { return M >= 3 || K > kDecodeMaxK; }

size_t gemv_workspace_bytes(int64_t M, int64_t K) {
    return M >= 1 && M <= kGemvMaxM && decode_on_tensor_cores(M, K) ? gemv_tc_workspace_bytes(M, K) : 0;
}

// The tensor-core decode puts the 128-row weight tiles in gridDim.y; the
// CUDA-core kernels cover any N (several launches when needed).
bool gemv_shape_supported(int64_t M, int64_t N, int64_t K) {
    return !decode_on_tensor_cores(M, K) || (N + 127) / 128 <= 65535;
}

namespace {
int sm_count_or_zero() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return device_sm_count(dev);
}
}  // namespace

// One row of x only: with two rows the grouped launches streamed slower than
// one launch per matrix (2943-2952 against 3194 GB/s for the four layer
// matrices), the two rows' x records leaving room for a shallower ring.
bool grouped_decode_eligible(int64_t M, int64_t N, int64_t K) {
    if (M != 1 || K % 1024 != 0 || decode_on_tensor_cores(M, K)) return false;
    const int sms = sm_count_or_zero();
    if (sms <= 0) return false;
    dp::GroupArgs a{};
    size_t smem = 0;
    int threads = 0;
    return dp::plan_group(1, sms, 1, &N, &K, a, smem, threads);
}

namespace {
// The next group from problem 0 of the arrays: as many problems (at most
// eight) as one launch's shared memory holds, with its plan; 0 when even the
// first does not fit.
int next_group(int G, int mt, int sms, const int64_t *N, const int64_t *K, dp::GroupArgs &a, size_t &smem,
               int &threads) {
    if (!dp::plan_group(mt, sms, 1, N, K, a, smem, threads)) return 0;
    int n = 1;
    while (n < G && n < dp::kMaxGroup) {
        dp::GroupArgs b{};
        size_t sm2 = 0;
        int th2 = 0;
        if (!dp::plan_group(mt, sms, n + 1, N, K, b, sm2, th2)) break;
        a = b;
        smem = sm2;
        threads = th2;
        ++n;
    }
    return n;
}
}  // namespace

int grouped_decode_launches(int G, int64_t M, const int64_t *N, const int64_t *K) {
    const int sms = sm_count_or_zero();
    if (sms <= 0 || M != 1) return -1;
    int launches = 0;
    for (int g0 = 0; g0 < G;) {
        dp::GroupArgs a{};
        size_t smem = 0;
        int threads = 0;
        const int n = next_group(G - g0, (int)M, sms, N + g0, K + g0, a, smem, threads);
        if (n == 0) return -1;
        ++launches;
        g0 += n;
    }
    return launches;
}

cudaError_t launch_gemv_grouped(int G, const uint16_t *const *x, const uint8_t *const *wq, float *const *y,
                                bool ybf16, int64_t M, const int64_t *N, const int64_t *K, cudaStream_t s,
                                unsigned int *err) {
    const int sms = sm_count_or_zero();
    if (sms <= 0) return cudaErrorInvalidDevice;
    if (M != 1) return cudaErrorInvalidValue;
    const int mt = 1;
    for (int g0 = 0; g0 < G;) {
        dp::GroupArgs a{};
        size_t smem = 0;
        int threads = 0;
        const int n = next_group(G - g0, mt, sms, N + g0, K + g0, a, smem, threads);
        if (n == 0) return cudaErrorInvalidValue;
        for (int g = 0; g < n; ++g) {
            a.it[g].x = x[g0 + g];
            a.it[g].wq = wq[g0 + g];
            a.it[g].y = y[g0 + g];
        }
        a.mrows = mt;
        a.ybf16 = ybf16 ? 1 : 0;
        const cudaError_t e = dp::launch_group<1>(a, smem, threads, sms, s, err);
        if (e != cudaSuccess) return e;
        g0 += n;
    }
    return cudaSuccess;
}

cudaError_t launch_gemv(const uint16_t *x, const uint8_t *wq, float *y, bool ybf16, int64_t M, int64_t N,
                        int64_t K, void *workspace, cudaStream_t s, unsigned int *err) {
    // three or more rows of x (or a K too long to hold in shared memory): the
    // dot product moves to the tensor cores
    if (decode_on_tensor_cores(M, K)) return launch_gemv_tc(x, wq, y, ybf16, M, N, K, workspace, s, err);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int sms = device_sm_count(dev);
    if (sms <= 0) return cudaErrorInvalidDevice;
    const int64_t rowbytes = K / 32 * 18;
    auto grid_for = [&](int64_t n) { return (int)(n < sms ? n : sms); };
    // the integer-dot kernel (both rows of x in one pass over the weights)
    const int mt_dp = (int)M;
    const int64_t ndp = rows_per_launch(N, [&](int64_t n) { return dp::fits(mt_dp, n, K, sms); });
    if (ndp > 0) {
        for (int64_t n0 = 0; n0 < N; n0 += ndp) {
            const int64_t n = N - n0 < ndp ? N - n0 : ndp;
            e = M == 1 ? dp::launch<1>(x, wq + n0 * rowbytes, y_offset(y, n0, ybf16), ybf16, n, N, K, sms, s, err)
                       : dp::launch<2>(x, wq + n0 * rowbytes, y_offset(y, n0, ybf16), ybf16, n, N, K, sms, s, err);
            if (e != cudaSuccess) return e;
        }
        return cudaSuccess;
    }
    // the binary16 kernel (K % 1024 != 0, or a K the integer kernel's
    // threads cannot cover): both rows of x per pass where they fit
    const int64_t ng =
        rows_per_launch(N, [&](int64_t n) { return plan_gemv(1, n, K, grid_for(n)).smem <= kSmemLimit; });
    if (ng == 0) return cudaErrorInvalidValue;
    for (int64_t n0 = 0; n0 < N; n0 += ng) {
        const int64_t n = N - n0 < ng ? N - n0 : ng;
        const int grid = grid_for(n);
        const int mt = M == 2 && plan_gemv(2, n, K, grid).smem <= kSmemLimit ? 2 : 1;
        for (int64_t m0 = 0; m0 < M; m0 += mt) {
            GemvPlan p = plan_gemv(mt, n, K, grid);
            p.args.mrows = (int)((M - m0) < mt ? (M - m0) : mt);
            p.args.ybf16 = ybf16 ? 1 : 0;
            p.args.ldy = N;
            const uint16_t *xm = x + m0 * K;
            float *ym = y_offset(y, m0 * N + n0, ybf16);
            e = mt == 1 ? launch_mt<1>(xm, wq + n0 * rowbytes, ym, p, grid, s, err)
                        : launch_mt<2>(xm, wq + n0 * rowbytes, ym, p, grid, s, err);
            if (e != cudaSuccess) return e;
        }
    }
    return cudaSuccess;
}

}  // namespace q4_0
