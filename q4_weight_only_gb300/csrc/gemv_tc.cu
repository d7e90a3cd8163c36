// gemv_tc.cu -- batched decode (3 <= M <= 64) on the 5th-generation tensor
// cores.
//
// "Vertical disaggregation: maximizing model throughput on heterogeneous
// silicon", section "Every cycle counts: custom kernels" lists batch decode
// (several sessions sharing one pass over the weights) among the Q4_0
// kernels.  With M rows of x, CUDA-core FMAs cannot keep up with the weight
// stream once M reaches a few rows, so the dot product moves to tcgen05:
//
//   * A = dequantised weights, 128 rows x 128 k per slot, in tensor memory
//     (binary16, d * (q - 8) rounded once), written by eight dequant warps;
//     one MMA-warp iteration issues the slot's eight MMAs (the issuing warp
//     shares its scheduler with the dequant warps, so fewer, larger
//     iterations keep it off the critical path);
//   * B = x: a small kernel first rounds x to binary16 once per call (each
//     row scaled by a power of two that the stores of y undo exactly), already
//     in the 128-byte-swizzled K-major tiles the MMA reads (rows >= M zero),
//     into a workspace of TM * K * 2 bytes; every CTA then brings in each
//     stage's x tile with one bulk copy.  Converting inside every CTA would
//     repeat the same work once per weight tile and load the schedulers of
//     two SM quarters more than the others;
//   * D = 128 x TM fp32 in tensor memory (TM = 16, 32 or 64, padded rows of x
//     are zero);
//   * N is tiled by 128 rows; when the tiles alone leave SMs idle, K is
//     split over S CTAs per tile, each streaming its K range once.  They
//     write their fp32 partial tiles to the workspace and count themselves
//     in on the tile's counter; the CTA that completes the count sums the S
//     partials in split order (deterministic; the only atomic is the integer
//     count) and writes y.  (Thread-block clusters with a distributed-shared-
//     memory reduction did the same without global scratch, but a grid of
//     7-CTA clusters took over 10 us to be dispatched onto the SMs.)
// Waits are bounded; every thread reaches the closing barriers even when a
// wait gives up.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <mutex>
#include <type_traits>

#include "q4_0_internal.h"
#include "q4_0_ptx.cuh"

namespace q4_0 {
namespace {

constexpr int kTileN = 128;               // weight rows per CTA (MMA M)
constexpr int kKB = 128;                  // k per A slot (one MMA-warp iteration: 8 MMAs)
constexpr int kKW = 256;                  // k per weight stage
constexpr int kSubs = kKW / kKB;          // A slots per weight stage
constexpr int kWRowBytes = kKW / 32 * 18;  // 144
constexpr int kWStageBytes = kTileN * kWRowBytes;
constexpr int kNA = 3;  // A slots: D + 3 x 64 TMEM columns <= 256
constexpr int kDequantWarps = 8;
constexpr int kThreads = 32 * (2 + kDequantWarps);  // 320

__host__ __device__ constexpr uint32_t cols_pow2(uint32_t v) {
    uint32_t p = 32;
    while (p < v) p <<= 1;
    return p;
}

// TM = 16 or 32: an x stage is one weight stage (256 k); TM = 64: an x
// stage is one A slot (128 k), so that three of them and the weight ring
// still leave room for a second CTA on the SM.
template <int TM>
struct Cfg {
    static constexpr uint32_t kXAtom = TM * 128;               // [TM x 64 k] fp16, 128-byte swizzle
    static constexpr int kXK = TM <= 32 ? kKW : kKB;           // k per x stage
    static constexpr int kSlotsPerX = kXK / kKB;               // A slots per x stage
    static constexpr uint32_t kXStage = kXAtom * (kXK / 64);
    static constexpr int kNX = TM <= 16 ? 4 : (TM <= 32 ? 2 : 3);  // x ring (two CTAs fit an SM)
    static constexpr int kNW = 3;  // weight ring (a fourth stage for 16- and 32-row tiles measured slower)
    static constexpr uint32_t kDCols = TM < 32 ? 32 : TM;
    static constexpr uint32_t kCols = cols_pow2(kDCols + kNA * (kKB / 2));
    static constexpr size_t kOffW = (size_t)kNX * kXStage;
    static constexpr size_t kOffBars = kOffW + (size_t)kNW * kWStageBytes;
    static constexpr int kNumBars = 2 * kNW + 2 * kNX + 2 * kNA + 3;
    static constexpr size_t kOffScale = kOffBars + ((kNumBars * 8 + 16 + 15) / 16) * 16;  // TM floats
    static constexpr size_t kSmem = 1024 + kOffScale + TM * 4;
};

__device__ __forceinline__ half2 u2h(uint32_t u) { return *reinterpret_cast<half2 *>(&u); }
__device__ __forceinline__ uint32_t h2u(half2 h) { return *reinterpret_cast<uint32_t *>(&h); }

// One Q4_0 block -> 16 TMEM columns of packed binary16 pairs, each value
// d * (q - 8) rounded once.  Exponent-bias decode with no nibble shifts: a
// low nibble OR-ed into the mantissa of 1024.0 gives 1024 + q, a high nibble
// masked in place gives 1024 + 16 q (both exact); (v - 1032) * d and
// (v - 1152) * (d / 16) are then exact small integers times d, rounded once.
// One 32-bit word of codes yields its bytes 0 and 2 (or 1 and 3) as a pair, so
// within every aligned group of four elements the pair order is (0, 2), (1, 3):
// k positions 1 and 2 of each group are swapped, and the x operand carries the
// same swap (swap_mid_pairs).  The shift by a byte is a high multiply, which
// runs on the FMA pipe rather than the ALU.
// kAnyScale false: d / 16 must be exact, i.e. |d| >= 2^-10 (scale_is_large);
// true: the high nibbles are shifted down and take the 1032 route too, which
// holds for every scale (subnormal and zero included) at two more
// instructions per word.  Both give the same bits.
__device__ __forceinline__ bool scale_is_large(uint32_t dbits) { return (dbits & 0x7C00u) >= 0x1400u; }

template <bool kAnyScale>
__device__ __forceinline__ void dequant_block16(uint32_t dbits, const uint32_t (&Q)[4], uint32_t (&out)[16],
                                                uint32_t kBias /* kNibbleBias, as a register */) {
    const half2 k1032 = u2h(0x64086408u), k1152 = u2h(0x64806480u);
    const half2 d2 = u2h(dbits * 0x00010001u);                  // (d, d)
    if (!kAnyScale) {
        const half2 d16 = __hmul2(d2, u2h(0x2C002C00u));         // d / 16, exact
#pragma unroll
        for (int wi = 0; wi < 4; ++wi) {
            const uint32_t q = Q[wi], t = __umulhi(q, 1u << 24);  // t = q >> 8
            out[2 * wi + 0] = h2u(__hmul2(__hsub2(u2h(and_or<0x000F000Fu>(q, kBias)), k1032), d2));
            out[2 * wi + 1] = h2u(__hmul2(__hsub2(u2h(and_or<0x000F000Fu>(t, kBias)), k1032), d2));
            out[8 + 2 * wi + 0] = h2u(__hmul2(__hsub2(u2h(and_or<0x00F000F0u>(q, kBias)), k1152), d16));
            out[8 + 2 * wi + 1] = h2u(__hmul2(__hsub2(u2h(and_or<0x00F000F0u>(t, kBias)), k1152), d16));
        }
        return;
    }
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
        const uint32_t q = Q[wi], t = q >> 8;
        out[2 * wi + 0] = h2u(__hmul2(__hsub2(u2h(and_or<0x000F000Fu>(q, kBias)), k1032), d2));
        out[2 * wi + 1] = h2u(__hmul2(__hsub2(u2h(and_or<0x000F000Fu>(t, kBias)), k1032), d2));
        out[8 + 2 * wi + 0] = h2u(__hmul2(__hsub2(u2h(and_or<0x000F000Fu>(q >> 4, kBias)), k1032), d2));
        out[8 + 2 * wi + 1] = h2u(__hmul2(__hsub2(u2h(and_or<0x000F000Fu>(t >> 4, kBias)), k1032), d2));
    }
}

// Swap the middle two binary16 values of each group of four held in the word
// pair (a, b) = (x0 x1, x2 x3) -> (x0 x2, x1 x3): the k order of the MMA's A
// tiles (see the dequantisation above).
__device__ __forceinline__ void swap_mid_pairs(uint32_t &a, uint32_t &b) {
    const uint32_t lo = __byte_perm(a, b, 0x5410), hi = __byte_perm(a, b, 0x7632);
    a = lo;
    b = hi;
}

// Largest magnitude among the eight bf16 values of a 16-byte chunk, as bits
// (for finite values the magnitude bits order like the magnitudes).
__device__ __forceinline__ uint32_t bf16x8_absmax_bits(uint4 u) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    uint32_t m = 0;
#pragma unroll
    for (int h = 0; h < 4; ++h) m = max(m, max(w[h] & 0x7FFFu, (w[h] >> 16) & 0x7FFFu));
    return m;
}

// x (bf16, [M][K]) -> the binary16 B tiles of gemv_tc_kernel, and zeroed
// split-K tile counters for it.  Each row is scaled by 2^shift so that its
// largest |x| lands in [2^14, 2^15) -- every element within 2^29 of it is a
// normal binary16 number and exact, none overflows, and tiny rows keep their
// precision -- and xscale[m] = 2^-shift (a power of two) is what the
// kernel's stores multiply by.  Stage u (256 k) is four atoms [TM rows x
// 64 k]; in an atom, row m is 128 bytes whose 16-byte chunk c sits at
// position c ^ (m & 7) (the 128-byte swizzle named in the MMA's shared-memory
// descriptor), values in the k order of the weight tiles; rows m >= M are
// zero.  One CTA per row of the tile: the row's maximum, then the
// conversion of the chunks the threads still hold in registers.  Rows of
// 8192 < K <= 24576 are first brought into shared memory by bulk copies
// (one round trip; with a thread's chunks beyond the eight it holds
// re-read from L2 in each pass, the down projection, K = 17408, took about
// 1 us longer per call); longer rows reload the rest.  128 threads of at
// most 56 registers, so that its CTAs fit beside two CTAs of the running
// decode kernel and start as soon as it completes (a staged row's 48 KB of
// shared memory at most still fits beside those of 16- and 32-row tiles,
// not beside 64-row ones).
constexpr int kXThreads = 128;
constexpr int kXHeld = 8;  // chunks per thread kept in registers between the passes (K <= 8192)
constexpr int kXStagedMaxK = 24576;  // rows staged in shared memory: K * 2 bytes <= 48 KB
__host__ __device__ constexpr bool x_row_staged(int64_t K) { return K > kXHeld * 8 * kXThreads && K <= kXStagedMaxK; }
template <int TM>
__global__ void __launch_bounds__(kXThreads, 9) x_tiles_kernel(const uint16_t *__restrict__ x, uint4 *__restrict__ xt,
                                                            float *__restrict__ xscale, int M, int K,
                                                            unsigned int *__restrict__ tile_cnt, int ncnt,
                                                            unsigned int *err) {
    extern __shared__ __align__(16) uint4 xrow[];  // the staged row (x_row_staged(K))
    __shared__ uint64_t xbar;
    __shared__ int xabort;
    pdl_launch_dependents();
    const int m = blockIdx.x;
    const int kc8 = K / 8;
    const uint4 *src = reinterpret_cast<const uint4 *>(x + (int64_t)m * K);
    const bool staged = x_row_staged(K);
    if (staged && threadIdx.x == 0) {
        mbar_init(&xbar, 1);
        xabort = 0;
        mbar_fence_init();
    }
    pdl_wait();  // x may come from the previous kernel (and the last one has read its counters)
    if (blockIdx.x == 0)  // the split-K tile counters of the matmul kernel that follows
        for (int i = threadIdx.x; i < ncnt; i += kXThreads) tile_cnt[i] = 0u;
    __shared__ uint32_t wmax[kXThreads / 32];
    uint4 held[kXHeld];
#pragma unroll
    for (int h = 0; h < kXHeld; ++h) held[h] = make_uint4(0, 0, 0, 0);
    uint32_t mb = 0;
    if (staged) {
        __syncthreads();  // the barrier's initialisation
        if (m < M) {
            if (threadIdx.x == 0) {
                const uint32_t bytes = (uint32_t)K * 2;
                mbar_arrive_expect_tx(&xbar, bytes);
                for (uint32_t off = 0; off < bytes; off += 16384)
                    bulk_g2s(reinterpret_cast<uint8_t *>(xrow) + off, reinterpret_cast<const uint8_t *>(src) + off,
                             bytes - off < 16384 ? bytes - off : 16384, &xbar);
            }
            const bool ok = mbar_wait(&xbar, 0, &xabort, err);
            for (int kc = threadIdx.x; ok && kc < kc8; kc += kXThreads) mb = max(mb, bf16x8_absmax_bits(xrow[kc]));
            if (!ok) mbar_drain(&xbar, 0);  // the copies land before the CTA can exit
        }
    } else if (m < M) {
#pragma unroll
        for (int h = 0; h < kXHeld; ++h) {
            const int kc = threadIdx.x + h * kXThreads;
            if (kc < kc8) {
                held[h] = __ldg(src + kc);
                mb = max(mb, bf16x8_absmax_bits(held[h]));
            }
        }
        for (int kc = threadIdx.x + kXHeld * kXThreads; kc < kc8; kc += kXThreads)
            mb = max(mb, bf16x8_absmax_bits(__ldg(src + kc)));
    }
    mb = __reduce_max_sync(0xffffffffu, mb);
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = mb;
    __syncthreads();
    mb = 0;
#pragma unroll
    for (int w = 0; w < kXThreads / 32; ++w) mb = max(mb, wmax[w]);
    int e = 0;
    if (mb != 0) frexpf(__uint_as_float(mb << 16), &e);  // max |x| in [2^(e-1), 2^e)
    const int shift = min(126, 15 - e);
    const float up = ldexpf(1.0f, shift);
    if (threadIdx.x == 0 && m < M) xscale[m] = ldexpf(1.0f, -shift);
    auto store = [&](int kc, uint4 u, bool live) {
        uint4 v = make_uint4(0, 0, 0, 0);
        if (live) {
            const uint32_t in[4] = {u.x, u.y, u.z, u.w};
            uint32_t o[4];
#pragma unroll
            for (int h = 0; h < 4; ++h)
                o[h] = h2u(__floats2half2_rn(__uint_as_float(in[h] << 16) * up,
                                             __uint_as_float(in[h] & 0xFFFF0000u) * up));
            swap_mid_pairs(o[0], o[1]);
            swap_mid_pairs(o[2], o[3]);
            v = make_uint4(o[0], o[1], o[2], o[3]);
        }
        const int u4 = kc >> 5, a = (kc >> 3) & 3, c = kc & 7;
        xt[((int64_t)(u4 * 4 + a) * TM + m) * 8 + (c ^ (m & 7))] = v;
    };
    if (staged) {
        for (int kc = threadIdx.x; kc < kc8; kc += kXThreads)
            store(kc, m < M ? xrow[kc] : make_uint4(0, 0, 0, 0), m < M);
        return;
    }
#pragma unroll
    for (int h = 0; h < kXHeld; ++h) {
        const int kc = threadIdx.x + h * kXThreads;
        if (kc < kc8) store(kc, held[h], m < M);
    }
    for (int kc = threadIdx.x + kXHeld * kXThreads; kc < kc8; kc += kXThreads)
        store(kc, m < M ? __ldg(src + kc) : make_uint4(0, 0, 0, 0), m < M);
}

template <int TM>
__global__ void __launch_bounds__(kThreads, 2)
    gemv_tc_kernel(const uint4 *__restrict__ xt, const __grid_constant__ CUtensorMap wmap,
                   float *__restrict__ y, float *__restrict__ part, unsigned int *__restrict__ tile_cnt,
                   const float *__restrict__ xscale, int M, int N, int K, int ybf16, uint32_t nib_bias,
                   unsigned int *err) {
    using C = Cfg<TM>;
    constexpr int kNX = C::kNX, kNW = C::kNW;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *xring = smem;
    uint8_t *wring = smem + C::kOffW;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBars);
    uint64_t *w_full = bars, *w_empty = bars + kNW;
    uint64_t *x_full = bars + 2 * kNW, *x_empty = x_full + kNX;
    uint64_t *a_full = x_empty + kNX, *a_empty = a_full + kNA;
    uint64_t *d_full = a_empty + kNA, *drain = d_full + 1, *s_full = drain + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + C::kNumBars);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    float *xs_smem = reinterpret_cast<float *>(smem + C::kOffScale);  // the x rows' scales [TM]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = gridDim.x;                 // CTAs per tile, along K
    const int rank = blockIdx.x;
    const int n0 = blockIdx.y * kTileN;
    const int KU = K / kKW;
    const int u0 = rank * KU / S, u1 = (rank + 1) * KU / S;
    const int nW = u1 - u0, nS = nW * kSubs;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kNW; ++i) {
            mbar_init(&w_full[i], 1);
            mbar_init(&w_empty[i], kDequantWarps);  // one arrival per warp
        }
        for (int i = 0; i < kNX; ++i) {
            mbar_init(&x_full[i], 1);
            mbar_init(&x_empty[i], 1);
        }
        for (int i = 0; i < kNA; ++i) {
            mbar_init(&a_full[i], kDequantWarps / 2);  // one half of the dequant warps
            mbar_init(&a_empty[i], 1);
        }
        mbar_init(d_full, 1);
        mbar_init(drain, 1);
        mbar_init(s_full, 1);
        *abort_flag = 0;
        mbar_fence_init();
        tma_prefetch_desc(&wmap);
    }
    if (warp == 1) tmem_alloc(tmem_slot, C::kCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_launch_dependents();
    const uint32_t tmem = *tmem_slot;
    const uint32_t d_tmem = tmem, a_tmem = tmem + C::kDCols;

    if (warp == 0) {
        if (lane == 0) {
            // copies: the first weight stages go out before the wait for the
            // previous kernel (weights do not depend on it); then, per stage,
            // its x tile and the weight stage kNW ahead
            const uint64_t policy = l2_evict_first_policy();  // weights are read once
            int issued_w = 0, issued_x = 0;
            auto issue_w = [&](int ws) -> bool {
                const int wsl = ws % kNW;
                if (!mbar_wait(&w_empty[wsl], ((ws / kNW) & 1) ^ 1, abort_flag, err)) return false;
                mbar_arrive_expect_tx(&w_full[wsl], kWStageBytes);
                tma_load_2d_hint(wring + wsl * kWStageBytes, &wmap, (u0 + ws) * kWRowBytes, n0, &w_full[wsl],
                                 policy);
                ++issued_w;
                return true;
            };
            // x stage xi of this CTA's K range (its tiles are contiguous in
            // the workspace: stage u of 256 k is four 64-k atoms)
            auto issue_x = [&](int xi) -> bool {
                const int xsl = xi % kNX;
                if (!mbar_wait(&x_empty[xsl], ((xi / kNX) & 1) ^ 1, abort_flag, err)) return false;
                mbar_arrive_expect_tx(&x_full[xsl], C::kXStage);
                bulk_g2s(xring + xsl * C::kXStage,
                         xt + ((size_t)u0 * (kKW / C::kXK) + xi) * (C::kXStage / 16), C::kXStage, &x_full[xsl]);
                ++issued_x;
                return true;
            };
            bool ok = true;
            for (int ws = 0; ok && ws < kNW && ws < nW; ++ws) ok = issue_w(ws);
            pdl_wait();  // the x tiles come from the previous kernel
            // the x rows' scales for the stores of y (the workspace holds room
            // for 64 of them, so the copy stays inside it for any M)
            mbar_arrive_expect_tx(s_full, TM * 4);
            bulk_g2s(xs_smem, xscale, TM * 4, s_full);
            for (int ws = 0; ok && ws < nW; ++ws) {
                for (int h = 0; ok && h < kKW / C::kXK; ++h) ok = issue_x(ws * (kKW / C::kXK) + h);
                if (ok && ws + kNW < nW) ok = issue_w(ws + kNW);
            }
            // let every issued copy land before the CTA can exit
            for (int i = issued_w - kNW; i < issued_w; ++i)
                if (i >= 0) mbar_drain(&w_full[i % kNW], (i / kNW) & 1);
            for (int i = issued_x - kNX; i < issued_x; ++i)
                if (i >= 0) mbar_drain(&x_full[i % kNX], (i / kNX) & 1);
            mbar_drain(s_full, 0);
        }
        __syncwarp();  // lanes 1..31 wait for the producer lane before the closing barriers
    } else if (warp == 1) {
        // MMA issue: the whole warp waits and loops (converged); one elected
        // lane issues the MMAs and commits
        constexpr uint32_t idesc = idesc_f16_f32(kTileN, TM);
        const uint64_t bdesc0 = smem_desc_k128(xring);
        // one A slot: wait for its x tile (first slot of a stage) and its
        // dequantised weights, issue its eight MMAs, release both.  x atoms of
        // 64 k are contiguous, so the descriptor's start address moves by one
        // atom every four MMAs.
        // sub: the slot's place in its x stage
        auto slot = [&](int s, int sub, int xsl, int asl, uint32_t xpar, uint32_t apar) -> bool {
            if (sub == 0 && !__all_sync(0xffffffffu, mbar_wait(&x_full[xsl], xpar, abort_flag, err))) return false;
            if (!__all_sync(0xffffffffu, mbar_wait(&a_full[asl], apar, abort_flag, err))) return false;
            tc_fence_after();
            if (elect_one()) {
                const uint64_t bdesc = bdesc0 + ((xsl * C::kXStage + sub * (kKB / 64) * C::kXAtom) >> 4);
#pragma unroll
                for (int kk = 0; kk < kKB / 16; ++kk)
                    mma_f16_ts(d_tmem, a_tmem + asl * (kKB / 2) + kk * 8,
                               bdesc + (kk / 4) * (C::kXAtom >> 4) + 2 * (kk % 4), idesc, (s | kk) != 0);
                mma_commit(&a_empty[asl]);
                if (sub == C::kSlotsPerX - 1) mma_commit(&x_empty[xsl]);
            }
            __syncwarp();
            return true;
        };
        bool ok = true;
        for (int s = 0; ok && s < nS; ++s) {
            const int xi = s / C::kSlotsPerX;
            ok = slot(s, s % C::kSlotsPerX, xi % kNX, s % kNA, (uint32_t)(xi / kNX) & 1u, (uint32_t)(s / kNA) & 1u);
        }
        if (elect_one()) mma_commit(d_full);
        __syncwarp();
    } else if (warp < 2 + kDequantWarps) {
        // dequant: warp (quarter q, half h) writes the A slot of k half h of
        // every weight stage (four blocks, 64 TMEM columns) for the 32 weight
        // rows of its lane quarter; one wait for both stores
        const int quad = warp & 3, half = (warp - 2) >> 2;
        const int r = quad * 32 + lane;
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        // ring slots and phases advance incrementally (A slot s = 2 ws + half
        // steps by two through a ring of three)
        auto dequant = [&]() -> bool {
            int wsl = 0, asl = half;
            uint32_t wph = 0, aph = 0;
            for (int ws = 0; ws < nW; ++ws) {
                if (!__all_sync(0xffffffffu, mbar_wait(&w_full[wsl], wph, abort_flag, err))) return false;
                // this warp's half of the row (bytes 72h .. 72h + 71) with nine
                // 8-byte loads: with a 144-byte row stride each load costs two
                // shared-memory wavefronts, as many as the 16-byte loads of the
                // same bytes would, and both halves run the same code
                const uint2 *row =
                    reinterpret_cast<const uint2 *>(wring + wsl * kWStageBytes + r * kWRowBytes + 72 * half);
                uint32_t rw[18];
#pragma unroll
                for (int i = 0; i < 9; ++i) {
                    const uint2 q = row[i];
                    rw[2 * i + 0] = q.x;
                    rw[2 * i + 1] = q.y;
                }
                // A slot (stage, half): 128 k = two 64-k pieces of 32 columns
                if (!__all_sync(0xffffffffu, mbar_wait(&a_empty[asl], aph ^ 1, abort_flag, err))) return false;
                tc_fence_after();
                // the route is chosen once for the warp's four blocks of the
                // stage: a branch per block cost about a tenth of the rate
                const bool large = scale_is_large(rw[0] & 0xFFFFu) && scale_is_large(rw[4] >> 16) &&
                                   scale_is_large(rw[9] & 0xFFFFu) && scale_is_large(rw[13] >> 16);
                auto slot_pieces = [&](auto any_c) {
                    constexpr bool kAny = decltype(any_c)::value;
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const uint32_t *wv = rw + 9 * j;
                        const uint32_t Q0[4] = {__funnelshift_r(wv[0], wv[1], 16), __funnelshift_r(wv[1], wv[2], 16),
                                                __funnelshift_r(wv[2], wv[3], 16), __funnelshift_r(wv[3], wv[4], 16)};
                        const uint32_t Q1[4] = {wv[5], wv[6], wv[7], wv[8]};
                        uint32_t cols[32];
                        uint32_t (&lo)[16] = *reinterpret_cast<uint32_t(*)[16]>(cols);
                        uint32_t (&hi)[16] = *reinterpret_cast<uint32_t(*)[16]>(cols + 16);
                        dequant_block16<kAny>(wv[0] & 0xFFFFu, Q0, lo, nib_bias);
                        dequant_block16<kAny>(wv[4] >> 16, Q1, hi, nib_bias);
                        tmem_st32(a_tmem + lane_base + asl * (kKB / 2) + j * 32, cols);
                    }
                };
                if (__all_sync(0xffffffffu, large))
                    slot_pieces(std::integral_constant<bool, false>{});
                else
                    slot_pieces(std::integral_constant<bool, true>{});
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();  // every lane's stores are done
                if (lane == 0) {
                    mbar_arrive(&a_full[asl]);
                    // the weight stage goes back only now that every lane has
                    // used what it loaded: a release right after the shared
                    // loads let the next TMA fill of the slot overtake loads
                    // still in flight (an async-proxy write after generic
                    // reads), seen as stale rows when weights came from L2
                    mbar_arrive(&w_empty[wsl]);
                }
                if (++wsl == kNW) {
                    wsl = 0;
                    wph ^= 1;
                }
                asl += kSubs;
                if (asl >= kNA) {
                    asl -= kNA;
                    aph ^= 1;
                }
            }
            return true;
        };
        static_assert(kSubs < kNA, "the A slot advances by kSubs and wraps at most once per stage");
        bool ok = dequant();
        // epilogue (warps 2..5 cover the four lane quarters): D -> partial tile
        if (half == 0) {
            if (ok) ok = __all_sync(0xffffffffu, mbar_wait(d_full, 0, abort_flag, err));
            // one K split stores y and needs the x rows' scales
            if (ok && S == 1) ok = __all_sync(0xffffffffu, mbar_wait(s_full, 0, abort_flag, err));
            if (ok) {
                tc_fence_after();
                uint32_t v[16];
                const int n = n0 + r;
                // one K split: y directly; else this split's partial tile,
                // [tile][split][m][128 rows] (coalesced over the rows)
                float *pt = part + ((size_t)blockIdx.y * S + rank) * TM * kTileN + r;
#pragma unroll
                for (int c = 0; c < TM; c += 16) {
                    tmem_ld16(d_tmem + lane_base + c, v);
                    tmem_wait_ld();
#pragma unroll
                    float sc[16];  // outside the store predicates: four 16-byte shared loads
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float4 t = reinterpret_cast<const float4 *>(xs_smem + c)[q];
                        sc[4 * q] = t.x;
                        sc[4 * q + 1] = t.y;
                        sc[4 * q + 2] = t.z;
                        sc[4 * q + 3] = t.w;
                    }
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int m = c + j;
                        if (m >= M) break;
                        if (S == 1) {
                            if (n < N) store_y(y, (int64_t)m * N + n, __uint_as_float(v[j]) * sc[j], ybf16 != 0);
                        } else {
                            pt[(size_t)m * kTileN] = __uint_as_float(v[j]);
                        }
                    }
                }
                if (S > 1) __threadfence();  // the partials before the count below
            }
        }
    }

    // split-K: count this CTA in; the CTA that completes the tile's count
    // sums the S partial tiles in split order and writes y
    __shared__ int last_s;
    __syncthreads();
    if (S > 1) {
        if (threadIdx.x == 0) last_s = atomicAdd(&tile_cnt[blockIdx.y], 1u) == (unsigned)(S - 1);
        __syncthreads();
        if (last_s) {
            __threadfence();
            // a thread sums groups of four rows of one x row (16-byte loads);
            // the partials of its two groups and of up to eight splits are
            // all in flight at once, so the sum costs one L2 round trip per
            // eight splits rather than one per element.  Each value is still
            // added in split order.
            const float4 *pt = reinterpret_cast<const float4 *>(part + (size_t)blockIdx.y * S * TM * kTileN);
            constexpr int kGroupsPerRow = kTileN / 4;
            constexpr size_t kSplitStride = (size_t)TM * kGroupsPerRow;  // float4s per partial tile
            const int groups = M * kGroupsPerRow;
            for (int g0 = threadIdx.x; g0 < groups; g0 += 2 * kThreads) {
                float4 sum[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) sum[h] = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int q0 = 0; q0 < S; q0 += 8) {
                    float4 v[2][8];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int g = g0 + h * kThreads;
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            v[h][q] = g < groups && q0 + q < S ? __ldcg(pt + (size_t)(q0 + q) * kSplitStride + g)
                                                               : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            sum[h].x += v[h][q].x;
                            sum[h].y += v[h][q].y;
                            sum[h].z += v[h][q].z;
                            sum[h].w += v[h][q].w;
                        }
                }
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int g = g0 + h * kThreads;
                    if (g >= groups) continue;
                    const int m = g / kGroupsPerRow, n = n0 + 4 * (g - m * kGroupsPerRow);
                    const float sc = __ldg(xscale + m);  // the x row's 2^-shift (exact)
                    const float s4[4] = {sum[h].x * sc, sum[h].y * sc, sum[h].z * sc, sum[h].w * sc};
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (n + j < N) store_y(y, (int64_t)m * N + n + j, s4[j], ybf16 != 0);
                }
            }
        }
    }
    if (warp == 1) {
        if (lane == 0) {
            mma_commit(drain);
            mbar_drain(drain, 0);
        }
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::kCols);
    }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Workspace: the x tiles, the x rows' scales, then room for 2 * SMs partial
// tiles (S * tiles never exceeds that when S > 1), then 2 * SMs tile
// counters.
struct WorkspaceLayout {
    size_t scale_off, part_off, cnt_off, bytes;
    WorkspaceLayout(int tm, int64_t K, int sms) {
        const size_t xt = (size_t)tm * (size_t)K * 2;
        scale_off = (xt + 255) / 256 * 256;
        part_off = scale_off + 256;  // tm <= 32 floats
        const size_t pb = (size_t)2 * (size_t)sms * kTileN * (size_t)tm * 4;
        cnt_off = part_off + pb;
        bytes = cnt_off + ((size_t)2 * (size_t)sms * 4 + 255) / 256 * 256 * (sms > 0 ? 1 : 0);
    }
};

template <int TM>
cudaError_t launch_tm(const uint16_t *x, const uint8_t *wq, float *y, bool ybf16, int64_t M, int64_t N,
                      int64_t K, void *workspace, cudaStream_t s, unsigned int *err) {
    using C = Cfg<TM>;
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    CUtensorMap wmap;
    {
        const cuuint64_t rowbytes = (cuuint64_t)(K / 32) * 18;
        const cuuint64_t dims[2] = {rowbytes, (cuuint64_t)N};
        const cuuint64_t strides[1] = {rowbytes};
        const cuuint32_t box[2] = {kWRowBytes, kTileN};
        const cuuint32_t estr[2] = {1, 1};
        if (enc(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(wq), dims, strides, box,
                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(gemv_tc_kernel<TM>), (int)C::kSmem);
    if (e != cudaSuccess) return e;
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int sms = device_sm_count(dev);
    const int64_t tiles = (N + kTileN - 1) / kTileN;
    const int64_t KU = K / kKW;
    // split K so that about two CTAs per SM are busy: S * tiles <= 2 * SMs,
    // which bounds the partial tiles the workspace holds
    int64_t S = tiles > 0 ? (2 * (int64_t)sms) / tiles : 1;
    S = S < 1 ? 1 : S;
    if (S > KU) S = KU;
    if (tiles > 65535 || S > 65535) return cudaErrorInvalidValue;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const WorkspaceLayout L(TM, K, sms);
    float *part = reinterpret_cast<float *>(ws + L.part_off);
    float *xscale = reinterpret_cast<float *>(ws + L.scale_off);
    unsigned int *cnt = reinterpret_cast<unsigned int *>(ws + L.cnt_off);
    e = launch_pdl(x_tiles_kernel<TM>, dim3((unsigned)TM), dim3(kXThreads), x_row_staged(K) ? (size_t)K * 2 : 0, s,
                   x, reinterpret_cast<uint4 *>(ws), xscale, (int)M, (int)K, cnt, S > 1 ? (int)tiles : 0, err);
    if (e != cudaSuccess) return e;
    return launch_pdl(gemv_tc_kernel<TM>, dim3((unsigned)S, (unsigned)tiles), dim3(kThreads), C::kSmem, s,
                      reinterpret_cast<const uint4 *>(ws), wmap, y, part, cnt, static_cast<const float *>(xscale),
                      (int)M, (int)N, (int)K, ybf16 ? 1 : 0, kNibbleBias, err);
}

}  // namespace

namespace {
int tile_rows_tc(int64_t M) { return M <= 16 ? 16 : (M <= 32 ? 32 : 64); }
}  // namespace

size_t gemv_tc_workspace_bytes(int64_t M, int64_t K) {
    int dev = 0;
    const int sms = cudaGetDevice(&dev) == cudaSuccess ? device_sm_count(dev) : 0;
    if (sms <= 0) (void)cudaGetLastError();
    return WorkspaceLayout(tile_rows_tc(M), K, sms > 0 ? sms : 0).bytes;
}

cudaError_t launch_gemv_tc(const uint16_t *x, const uint8_t *wq, float *y, bool ybf16, int64_t M, int64_t N,
                           int64_t K, void *workspace, cudaStream_t s, unsigned int *err) {
    switch (tile_rows_tc(M)) {
        case 16: return launch_tm<16>(x, wq, y, ybf16, M, N, K, workspace, s, err);
        case 32: return launch_tm<32>(x, wq, y, ybf16, M, N, K, workspace, s, err);
        default: return launch_tm<64>(x, wq, y, ybf16, M, N, K, workspace, s, err);
    }
}

}  // namespace q4_0
