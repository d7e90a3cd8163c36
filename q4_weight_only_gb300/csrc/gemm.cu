// gemm.cu -- prefill GEMM y = x * W^T on the 5th-generation tensor cores.
//
// "Vertical disaggregation: maximizing model throughput on heterogeneous
// silicon", section "Every cycle counts: custom kernels" names a GPU
// "Q4_0 -> Tensor Core" path over the shared Q4_0 format.  On sm_103a:
//
//   * x (bf16) is first rounded to binary16 into a scratch buffer, because a
//     tcgen05 kind::f16 MMA takes A and B of one type and binary16 operand
//     tiles keep the result well inside the error budget (bf16 weight tiles
//     would not); each row of x is scaled by a power of two first (its
//     largest |x| into [2^14, 2^15)), which the epilogue undoes exactly, so
//     any finite bf16 row fits binary16's range;
//   * one CTA computes a 128 (weight rows) x TM (x rows) tile of y^T, TM a
//     multiple of 16 chosen per call: the fewest tiles of at most 320 rows
//     (every further tile dequantises each weight tile again; M = 272 is one
//     tile, not two of 144), with the least padding.  Past 256 rows an x
//     stage arrives as two TMA boxes and each k step takes a second MMA for
//     rows 256.. (an MMA is at most 256 wide);
//     warp 0 streams Q4_0 weight tiles [128 rows x 256 k] (144 bytes per row)
//     and 128-byte-swizzled x tiles [TM rows x 64 k] with tensor TMA;
//   * warps 2-5 (one thread per weight row) unpack nibbles, apply the scale
//     in binary16 (d * (q - 8), one rounding) and store the tile into tensor
//     memory with tcgen05.st -- the A operand of the MMA lives in TMEM, so
//     dequantised weights never touch shared memory;
//   * warp 1 issues tcgen05.mma (M = 128, N = TM, K = 16) with A from TMEM,
//     B from shared memory, fp32 accumulation in TMEM;
//   * warps 2-5 then read the accumulator with tcgen05.ld and store y with
//     32 consecutive n per warp store (coalesced).
// All pipeline waits are bounded (see q4_0_ptx.cuh); the reduction order is
// fixed, so results are deterministic.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <mutex>
#include <type_traits>

#include "q4_0_internal.h"
#include "q4_0_ptx.cuh"

namespace q4_0 {
namespace {

constexpr int kTileN = 128;                 // weight rows per CTA (MMA M)
constexpr int kKW = 256;                    // k per weight stage
constexpr int kWRowBytes = kKW / 32 * 18;   // 144
constexpr int kWStageBytes = kTileN * kWRowBytes;
constexpr int kNW = 3;                      // weight ring depth
// A slot and x stage: 128 k for tiles of 129..192 rows and tall tiles, 64 k
// otherwise.  Every slot costs the MMA warp two barrier waits, two commits
// and a fence, about as long as the four MMAs of a 64-k slot for 256 x rows;
// a 128-k slot (eight MMAs) leaves the tensor pipe the longer of the two.
// Tiles of 193..256 rows keep 64 k: two 128-k stages of x (all that fits)
// hold less x in flight than five 64-k ones, and measured slower.  Small
// tiles keep 64 k too (their CTAs pair up on an SM, which halves the tensor
// memory and shared memory a CTA may hold).
constexpr int kWideSlotMinRows = 129, kWideSlotMaxRows = 192;
constexpr int kMaxTileRowsShort = 256;      // one MMA wide; taller tiles take a second MMA
constexpr int kNAMax = 4;                   // A slots at most (fewer where tensor memory is short)
// x ring depth: two 128-k stages for tall tiles (up to 80 KB a stage), three
// for 129..192 rows (up to 48 KB); five 64-k stages for tiles of 193..256
// rows (32 KB) and for small tiles alone on an SM
constexpr int kNXShort = 5, kNXMid = 3, kNXTall = 2;
// Tiles of 96..128 rows keep two CTAs on an SM (twice the dequantising warps,
// which bind the GEMM at small M) only with a three-stage x ring; up to 80
// rows five stages fit beside a second CTA.
constexpr int kNXPair = 3, kPairMaxRows = 128;
// x tiles per band of the tile order (see gemm_kernel)
constexpr int kBandMTiles = 8;
constexpr int kMaxTileRows = 320;
// warp 0: weight copies; warp 1: MMA issue; warps 2-5: dequantisation and
// the epilogue; warps 6 and 7: x copies (even and odd stages of an even
// ring; an odd ring has one producer).  Issuing a bulk tensor copy holds the
// thread for about 0.15 us, so one thread issuing every copy fell behind the
// MMAs.
constexpr int kThreads = 256;
constexpr int kXProducerWarp = 6;

__host__ __device__ constexpr uint32_t pow2_at_least(uint32_t v) {
    uint32_t p = 32;
    while (p < v) p <<= 1;
    return p;
}

// k per A slot and x stage for a tile of tm rows.
__host__ __device__ constexpr int slot_k(int tm) { return tm >= kWideSlotMinRows ? 128 : 64; }
// k per x stage: 128 where the ring holds two or three such stages (tall
// tiles, 129..192 rows); tiles of 193..256 rows take their x in five 64-k
// chunks, two per A slot, so that the ring keeps as much x in flight as
// with 64-k slots
__host__ __device__ constexpr int xstage_k(int tm) {
    return tm > kMaxTileRowsShort || (tm >= kWideSlotMinRows && tm <= kWideSlotMaxRows) ? 128 : 64;
}

// Shared-memory and TMEM layout of a CTA for an x tile of `tm` rows: an x
// stage is slot_k / 64 chunks of [tm rows x 64 k] (128-byte rows, the MMA's
// 128-byte swizzle); an A slot slot_k / 2 TMEM columns.  Tiles of up to 128
// rows keep to 256 columns (two CTAs may share the SM's 512).
struct GemmLayout {
    uint32_t x_stage, d_cols, cols;
    size_t bar_off, scale_off, smem;
    int num_bars, na;
    __host__ __device__ GemmLayout(int tm, int nx) {
        const int sk = slot_k(tm);
        x_stage = (uint32_t)tm * 2 * xstage_k(tm);
        d_cols = tm < 32 ? 32 : (uint32_t)((tm + 31) / 32 * 32);
        const int budget = d_cols <= 128 ? 256 : 512;
        na = (budget - (int)d_cols) / (sk / 2) < kNAMax ? (budget - (int)d_cols) / (sk / 2) : kNAMax;
        cols = pow2_at_least(d_cols + na * (sk / 2));
        bar_off = (size_t)nx * x_stage + (size_t)kNW * kWStageBytes;
        num_bars = 2 * kNW + 2 * nx + 2 * kNAMax + 3;
        // the tile's x-row scales (tm rounded up to 32 floats), read as float4:
        // 16-byte aligned whatever the barrier count
        scale_off = (bar_off + num_bars * 8 + 16 + 15) / 16 * 16;
        smem = 1024 + scale_off + 2 * (size_t)((tm + 31) / 32 * 32) * 4;  // two scale buffers (persistent form)
    }
};

// The persistent form runs the tiles with 128-k A slots (more than 128
// rows, one CTA per SM) when there are more work units (tiles times K
// splits) than SMs, so that some CTA takes two or more.
bool use_persistent(int tm, int nx, int64_t tiles, int splits, int sms) {
    return slot_k(tm) == 128 && (nx == kNXShort || nx == kNXMid || nx == kNXTall) && sms > 0 &&
           tiles * splits > (int64_t)sms;
}

// x ring depth for a tile of tm rows when the launch has `ctas` CTAs on
// `sms` SMs: the shallow ring where it lets a second CTA share the SM
// (shared memory and tensor memory both fit two) and there are more CTAs
// than SMs to pair up; a CTA alone on its SM keeps the deep ring.
int x_ring_stages(int tm, int64_t ctas, int sms) {
    if (tm > kMaxTileRowsShort) return kNXTall;
    if (tm > kWideSlotMaxRows) return kNXShort;  // five 64-k chunks
    if (tm >= kWideSlotMinRows) return kNXMid;
    if (tm > 80 && tm <= kPairMaxRows && ctas > sms) return kNXPair;
    return kNXShort;
}

__device__ __forceinline__ half2 u2h(uint32_t u) { return *reinterpret_cast<half2 *>(&u); }
__device__ __forceinline__ uint32_t h2u(half2 h) { return *reinterpret_cast<uint32_t *>(&h); }

// Swap the middle two binary16 values of each group of four held in the word
// pair (a, b) = (x0 x1, x2 x3) -> (x0 x2, x1 x3): the k order of the MMA's A
// tiles (see dequant_block below).
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

// One row of x (bf16) -> binary16, scaled by 2^shift so that the row's
// largest |x| lands in [2^14, 2^15): every element within 2^29 of it is then
// a normal binary16 number and exact (bf16 has 8 significant bits), none
// overflows, and tiny rows keep their precision.  xscale[m] = 2^-shift is
// what the epilogue multiplies the fp32 accumulator by (exact: a power of
// two).  Values are written in the k order of the weight tiles (middle pair
// of every group of four swapped).  One CTA per row: the row's maximum, then
// the conversion of the chunks the threads still hold in registers (kHeld
// 16-byte chunks a thread; longer rows reload the rest in each pass).  The
// three-chunk form (K <= 6144) is small in registers, so that several CTAs
// fit beside the running GEMM's and start as soon as it completes; rows of
// 6144 < K <= 18432 take the nine-chunk form (64 registers, still one CTA
// beside the GEMM): re-reading a thread's chunks beyond the third in both
// passes had made the down projection (K = 17408) 2.4 us (M = 2048) to
// 3 us (M = 272) slower per call.
constexpr int kXThreads = 256;
constexpr int kXHeldShort = 3, kXHeldLong = 9;  // chunks held a thread: K <= 6144, K <= 18432
template <int kXHeld>
__global__ void __launch_bounds__(kXThreads, kXHeld <= 3 ? 8 : 4)
    x_to_f16_kernel(const uint4 *__restrict__ x, uint4 *__restrict__ x16, float *__restrict__ xscale, int kc8) {
    pdl_launch_dependents();
    pdl_wait();
    __shared__ uint32_t wmax[kXThreads / 32];
    const int64_t base = (int64_t)blockIdx.x * kc8;
    uint4 held[kXHeld];
    uint32_t mb = 0;
#pragma unroll
    for (int h = 0; h < kXHeld; ++h) {
        const int i = threadIdx.x + h * kXThreads;
        if (i < kc8) {
            held[h] = __ldg(x + base + i);
            mb = max(mb, bf16x8_absmax_bits(held[h]));
        }
    }
    for (int i = threadIdx.x + kXHeld * kXThreads; i < kc8; i += kXThreads)
        mb = max(mb, bf16x8_absmax_bits(__ldg(x + base + i)));
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
    if (threadIdx.x == 0) xscale[blockIdx.x] = ldexpf(1.0f, -shift);
    auto convert = [&](uint4 u) {
        const uint32_t in[4] = {u.x, u.y, u.z, u.w};
        uint32_t out[4];
#pragma unroll
        for (int h = 0; h < 4; ++h)
            out[h] = h2u(__floats2half2_rn(__uint_as_float(in[h] << 16) * up,
                                           __uint_as_float(in[h] & 0xFFFF0000u) * up));
        swap_mid_pairs(out[0], out[1]);
        swap_mid_pairs(out[2], out[3]);
        return make_uint4(out[0], out[1], out[2], out[3]);
    };
#pragma unroll
    for (int h = 0; h < kXHeld; ++h) {
        const int i = threadIdx.x + h * kXThreads;
        if (i < kc8) x16[base + i] = convert(held[h]);
    }
    for (int i = threadIdx.x + kXHeld * kXThreads; i < kc8; i += kXThreads) x16[base + i] = convert(__ldg(x + base + i));
}

// y = sum over splits of the partial tiles, in split order (deterministic);
// y is fp32, or bfloat16 rounded to nearest even when ybf16.  A thread's
// loads of all splits (at most four) are issued before the first add, so
// it pays one L2 round trip rather than one per split.
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float4 *__restrict__ part, float *__restrict__ y,
                                                            int64_t n4, int splits, int ybf16) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n4) return;
    float4 v[4];
#pragma unroll
    for (int z = 0; z < 4; ++z) v[z] = z < splits ? __ldcg(part + (int64_t)z * n4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    float4 acc = v[0];
#pragma unroll
    for (int z = 1; z < 4; ++z) {
        if (z >= splits) break;
        acc.x += v[z].x;
        acc.y += v[z].y;
        acc.z += v[z].z;
        acc.w += v[z].w;
    }
    if (ybf16) {
        const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
        reinterpret_cast<uint2 *>(y)[i] =
            make_uint2(*reinterpret_cast<const uint32_t *>(&lo), *reinterpret_cast<const uint32_t *>(&hi));
    } else {
        reinterpret_cast<float4 *>(y)[i] = acc;
    }
}

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
__device__ __forceinline__ void dequant_block(uint32_t dbits, const uint32_t (&Q)[4], uint32_t *out,
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

// Tile b of the launch order -> its first weight row n0 and x row m0.  Tiles
// come in bands of up to kBandMTiles x tiles; within a band, the x tiles of
// one weight tile are neighbours, so a weight tile comes from HBM once per
// band while the band's x rows stay in L2.
__device__ __forceinline__ void tile_origin(int64_t b, int NT, int MT, int TM, int &n0, int &m0) {
    const int64_t per_band = (int64_t)NT * kBandMTiles;
    const int bands = (MT + kBandMTiles - 1) / kBandMTiles;
    const int band = (int)(b / per_band < bands - 1 ? b / per_band : bands - 1);
    const int64_t r = b - (int64_t)band * per_band;
    const int gm = MT - band * kBandMTiles < kBandMTiles ? MT - band * kBandMTiles : kBandMTiles;
    n0 = (int)(r / gm) * kTileN;
    m0 = (band * kBandMTiles + (int)(r % gm)) * TM;
}

// kTall: x tiles of more than 256 rows (two TMA boxes per x chunk, a second
// MMA per k step); a separate instantiation keeps the common path unchanged.
// kNX: stages of the x ring.  kSK: k per A slot and x stage (slot_k(TM)).
template <bool kTall, int kNX, int kSK, int kXK>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap,
                float *__restrict__ y, float *__restrict__ part, const float *__restrict__ xscale, int M, int N,
                int K, int TM, int ybf16, uint32_t nib_bias, unsigned int *err) {
    constexpr int kChunks = kSK / 64;         // 64-k pieces per slot (A stores)
    constexpr int kXPerSlot = kSK / kXK;      // x stages per A slot
    constexpr int kXChunks = kXK / 64;        // 64-k chunks (TMA boxes) per x stage
    constexpr int kSlotsPerW = kKW / kSK;     // A slots per weight stage
    constexpr int kSlotCols = kSK / 2;        // TMEM columns per A slot
    const GemmLayout Cfg(TM, kNX);
    const int na = Cfg.na;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *xring = smem;
    uint8_t *wring = smem + kNX * Cfg.x_stage;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg.bar_off);
    uint64_t *w_full = bars, *w_empty = bars + kNW;
    uint64_t *x_full = bars + 2 * kNW, *x_empty = x_full + kNX;
    uint64_t *a_full = x_empty + kNX, *a_empty = a_full + kNAMax;
    uint64_t *d_full = a_empty + kNAMax, *drain = d_full + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + Cfg.num_bars);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    float *xs_tile = reinterpret_cast<float *>(smem + Cfg.scale_off);  // [TM]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NT = (N + kTileN - 1) / kTileN, MT = (M + TM - 1) / TM;
    int n0, m0;
    tile_origin(blockIdx.x, NT, MT, TM, n0, m0);
    // split-K: CTA z of gridDim.z takes weight stages [w_begin, w_end) and,
    // when split, writes its partial tile to part[z] instead of y
    const int KW_all = K / kKW;
    const int w_begin = (int)((int64_t)blockIdx.z * KW_all / gridDim.z);
    const int w_end = (int)((int64_t)(blockIdx.z + 1) * KW_all / gridDim.z);
    const int KWS = w_end - w_begin, KS = KWS * kSlotsPerW;
    float *out = part ? part + (size_t)blockIdx.z * M * N : nullptr;  // fp32 partial tile of a K split

    if (threadIdx.x == 0) {
        for (int i = 0; i < kNW; ++i) {
            mbar_init(&w_full[i], 1);
            mbar_init(&w_empty[i], 4);  // one arrival per dequant warp
        }
        for (int i = 0; i < kNX; ++i) {
            mbar_init(&x_full[i], 1);
            mbar_init(&x_empty[i], 1);
        }
        for (int i = 0; i < na; ++i) {
            mbar_init(&a_full[i], 4);
            mbar_init(&a_empty[i], 1);
        }
        mbar_init(d_full, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        mbar_fence_init();
        tma_prefetch_desc(&xmap);
        tma_prefetch_desc(&wmap);
    }
    if (warp == 1) tmem_alloc(tmem_slot, Cfg.cols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_launch_dependents();
    pdl_wait();  // x16 comes from the previous kernel
    const uint32_t tmem = *tmem_slot;
    const uint32_t d_tmem = tmem;
    const uint32_t a_tmem = tmem + Cfg.d_cols;

    if (warp == 0) {
        if (lane == 0) {
            // weight stages
            int issued_w = 0;
            for (int ws = 0; ws < KWS; ++ws) {
                const int wsl = ws % kNW;
                if (!mbar_wait(&w_empty[wsl], ((ws / kNW) & 1) ^ 1, abort_flag, err)) break;
                mbar_arrive_expect_tx(&w_full[wsl], kWStageBytes);
                tma_load_2d(wring + wsl * kWStageBytes, &wmap, (w_begin + ws) * kWRowBytes, n0, &w_full[wsl]);
                ++issued_w;
            }
            // let every issued copy land before the CTA can exit
            for (int i = issued_w - kNW; i < issued_w; ++i)
                if (i >= 0) mbar_drain(&w_full[i % kNW], (i / kNW) & 1);
        }
    } else if (warp == kXProducerWarp || warp == kXProducerWarp + 1) {
        // x stages: producer p takes stages p, p + P, ... (with an even ring
        // each producer owns its slots, so their phases follow in order)
        constexpr int P = kNX % 2 == 0 ? 2 : 1;
        const int p = warp - kXProducerWarp;
        if (lane == 0 && p < P) {
            const int KX = KS * kXPerSlot;  // x stages of this CTA's K range
            int next = p;  // first stage not issued
            for (int s = p; s < KX; s += P) {
                const int xsl = s % kNX;
                if (!mbar_wait(&x_empty[xsl], ((s / kNX) & 1) ^ 1, abort_flag, err)) break;
                mbar_arrive_expect_tx(&x_full[xsl], Cfg.x_stage);
                uint8_t *dst = xring + xsl * Cfg.x_stage;
#pragma unroll
                for (int j = 0; j < kXChunks; ++j) {
                    const int kx = w_begin * kKW + s * kXK + 64 * j;
                    tma_load_2d(dst + j * TM * 128, &xmap, kx, m0, &x_full[xsl]);
                    if (kTall)  // a TMA box is at most 256 rows: two boxes of TM / 2
                        tma_load_2d(dst + j * TM * 128 + (TM / 2) * 128, &xmap, kx, m0 + TM / 2, &x_full[xsl]);
                }
                next = s + P;
            }
            // let this producer's copies land before the CTA can exit
            for (int i = next - kNX; i < next; i += P)
                if (i >= 0) mbar_drain(&x_full[i % kNX], (i / kNX) & 1);
        }
    } else if (warp == 1) {
        // MMA issue: the whole warp waits and loops (converged); one elected
        // lane issues the MMAs and commits
        // an MMA is at most 256 wide: a taller x tile takes a second MMA per
        // k step over rows 256.. (D columns 256..), with the same A
        const uint32_t idesc = idesc_f16_f32(kTileN, (uint32_t)(kTall ? 256 : TM));
        const uint32_t idesc2 = idesc_f16_f32(kTileN, (uint32_t)(kTall ? TM - 256 : 16));
        int asl = 0;  // A slot s % na and its phase, advanced per slot (no runtime division)
        uint32_t aph = 0;
        bool ok = true;
        for (int s = 0; ok && s < KS; ++s) {
            // the slot's x stages g = s * kXPerSlot + u
#pragma unroll
            for (int u = 0; u < kXPerSlot; ++u) {
                const int g = s * kXPerSlot + u;
                ok = __all_sync(0xffffffffu, mbar_wait(&x_full[g % kNX], (g / kNX) & 1, abort_flag, err));
                if (!ok) break;
            }
            if (!ok) break;
            if (!__all_sync(0xffffffffu, mbar_wait(&a_full[asl], aph, abort_flag, err))) break;
            tc_fence_after();
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < kSK / 16; ++kk) {
                    // 64-k chunk kk / 4 of the slot: x stage u, chunk jj of it;
                    // a K = 16 step is 32 bytes along its rows
                    const int chunk = kk >> 2, u = chunk / kXChunks, jj = chunk % kXChunks;
                    const int g = s * kXPerSlot + u;
                    const uint64_t bdesc =
                        smem_desc_k128(xring + (g % kNX) * Cfg.x_stage + jj * TM * 128) + 2 * (kk & 3);
                    const uint32_t acol = a_tmem + asl * kSlotCols + kk * 8;
                    mma_f16_ts(d_tmem, acol, bdesc, idesc, (s | kk) != 0);
                    if (kTall)  // rows 256.. start 256 x 128 bytes into the chunk
                        mma_f16_ts(d_tmem + 256, acol, bdesc + (256 * 128 >> 4), idesc2, (s | kk) != 0);
                }
#pragma unroll
                for (int u = 0; u < kXPerSlot; ++u) mma_commit(&x_empty[(s * kXPerSlot + u) % kNX]);
                mma_commit(&a_empty[asl]);
            }
            __syncwarp();
            if (++asl == na) {
                asl = 0;
                aph ^= 1;
            }
        }
        if (elect_one()) mma_commit(d_full);
        __syncwarp();
    } else if (warp >= 2 && warp < 6) {
        // warps 2..5: dequantise into TMEM, then the epilogue
        const int quad = warp & 3;
        const int r = quad * 32 + lane;  // weight row within the tile
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        // the tile's x-row scales: loaded now (in flight during the mainloop),
        // put into shared memory for the epilogue after it -- loaded in the
        // epilogue, each would wait behind the tensor-memory loads and the
        // stores before it
        float sv[(kMaxTileRows + 127) / 128];
#pragma unroll
        for (int t = 0; t < (kMaxTileRows + 127) / 128; ++t) {
            const int i = threadIdx.x - 64 + 128 * t;
            sv[t] = i < TM && m0 + i < M ? __ldg(xscale + m0 + i) : 0.f;
        }
        bool ok = true;
        int asl = 0;  // A slot and its phase, advanced per slot
        uint32_t aph = 0;
        for (int ws = 0; ws < KWS && ok; ++ws) {
            const int wsl = ws % kNW;
            ok = __all_sync(0xffffffffu, mbar_wait(&w_full[wsl], (ws / kNW) & 1, abort_flag, err));
            if (!ok) break;
            // the row's 144 bytes with nine 16-byte loads: with a 144-byte row
            // stride the eight lanes of each load phase hit distinct 16-byte
            // bank groups (4-byte loads would conflict four ways).  The stage
            // goes back to the producer once every lane has used its row (after
            // the last slot): the next TMA fill of the slot is an async-proxy
            // write and must not overtake shared loads in flight.
            const uint4 *row = reinterpret_cast<const uint4 *>(wring + wsl * kWStageBytes + r * kWRowBytes);
            uint32_t rw[36];
#pragma unroll
            for (int i = 0; i < 9; ++i) {
                const uint4 q = row[i];
                rw[4 * i + 0] = q.x;
                rw[4 * i + 1] = q.y;
                rw[4 * i + 2] = q.z;
                rw[4 * i + 3] = q.w;
            }
            // the route is chosen once for the warp's eight blocks of the
            // stage: a branch per block cost about a tenth of the rate
            bool large = true;
#pragma unroll
            for (int q = 0; q < kKW / 64; ++q)
                large = large && scale_is_large(rw[9 * q] & 0xFFFFu) && scale_is_large(rw[9 * q + 4] >> 16);
            auto stage_slots = [&](auto any_c) {
                constexpr bool kAny = decltype(any_c)::value;
#pragma unroll
                for (int sub = 0; sub < kSlotsPerW; ++sub) {
                    ok = __all_sync(0xffffffffu, mbar_wait(&a_empty[asl], aph ^ 1, abort_flag, err));
                    if (!ok) break;
                    tc_fence_after();
                    // the slot's 64-k pieces: two blocks, 32 TMEM columns each
#pragma unroll
                    for (int pc = 0; pc < kChunks; ++pc) {
                        const uint32_t *wv = rw + 9 * (sub * kChunks + pc);
                        const uint32_t Q0[4] = {__funnelshift_r(wv[0], wv[1], 16),
                                                __funnelshift_r(wv[1], wv[2], 16),
                                                __funnelshift_r(wv[2], wv[3], 16),
                                                __funnelshift_r(wv[3], wv[4], 16)};
                        const uint32_t Q1[4] = {wv[5], wv[6], wv[7], wv[8]};
                        uint32_t cols[32];
                        dequant_block<kAny>(wv[0] & 0xFFFFu, Q0, cols, nib_bias);
                        dequant_block<kAny>(wv[4] >> 16, Q1, cols + 16, nib_bias);
                        tmem_st32(a_tmem + lane_base + asl * kSlotCols + pc * 32, cols);
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();  // every lane's stores are done
                    if (lane == 0) mbar_arrive(&a_full[asl]);
                    if (++asl == na) {
                        asl = 0;
                        aph ^= 1;
                    }
                }
            };
            if (__all_sync(0xffffffffu, large))
                stage_slots(std::integral_constant<bool, false>{});
            else
                stage_slots(std::integral_constant<bool, true>{});
            if (lane == 0) mbar_arrive(&w_empty[wsl]);
        }
        // epilogue: D[row r][column m] -> y[m][n0 + r], times the x row's
        // scale 2^-shift (a power of two, so a K split's partial tiles sum
        // to the same bits as the unsplit tile)
#pragma unroll
        for (int t = 0; t < (kMaxTileRows + 127) / 128; ++t) {
            const int i = threadIdx.x - 64 + 128 * t;
            if (i < (TM + 31) / 32 * 32) xs_tile[i] = sv[t];
        }
        named_bar_sync(1, 128);  // the four epilogue warps
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(d_full, 0, abort_flag, err));
        if (ok) {
            tc_fence_after();
            const int n = n0 + r;
            for (int c = 0; c < TM; c += 32) {
                uint32_t v[32];
                tmem_ld32(d_tmem + lane_base + c, v);
                // the 32 scales of these columns: eight 16-byte shared loads,
                // outside the store predicates
                float sc[32];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 t = reinterpret_cast<const float4 *>(xs_tile + c)[q];
                    sc[4 * q] = t.x;
                    sc[4 * q + 1] = t.y;
                    sc[4 * q + 2] = t.z;
                    sc[4 * q + 3] = t.w;
                }
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int m = m0 + c + j;
                    const float val = __uint_as_float(v[j]) * sc[j];
                    if (c + j < TM && m < M && n < N) {
                        if (out)
                            out[(int64_t)m * N + n] = val;
                        else
                            store_y(y, (int64_t)m * N + n, val, ybf16 != 0);
                    }
                }
            }
        }
    }
    __syncthreads();
    if (warp == 1) {
        if (lane == 0) {
            // every MMA issued by this CTA has finished before TMEM is released
            mma_commit(drain);
            mbar_drain(drain, 0);
        }
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, Cfg.cols);
    }
}

// Persistent form of gemm_kernel for tiles of one MMA width fed by 64-k x
// chunks, when there are at least two tiles per SM and no K split: one CTA
// per SM takes tiles u = c, c + G, ... of the band order.  Four extra warps
// run the epilogue, so that while they store tile i the producers and the
// dequantising warps already work on tile i + 1 (its copies land and its
// first A slots fill); the MMAs of tile i + 1 start once the epilogue has
// read the accumulator.  One-tile-per-CTA launches paid the CTA's start,
// its pipeline fill and the gap to the next CTA on every tile.
// Warps: 0 weight copies, 1 MMA issue, 2-5 dequantisation, 6 x copies
// (7 idle), 8-11 epilogue.
constexpr int kPThreads = 384;
constexpr int kPEpiWarp0 = 8;

template <bool kTall, int kNX, int kSK, int kXK>
__global__ void __launch_bounds__(kPThreads, 1)
    gemm_persistent_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap,
                           float *__restrict__ y, float *__restrict__ part, const float *__restrict__ xscale, int M,
                           int N, int K, int TM, int splits, int ybf16, uint32_t nib_bias,
                           unsigned int *err) {
    constexpr int kChunks = kSK / 64;
    constexpr int kXPerSlot = kSK / kXK;
    constexpr int kXChunks = kXK / 64;
    constexpr int kSlotsPerW = kKW / kSK;
    constexpr int kSlotCols = kSK / 2;
    constexpr int P = kNX % 2 == 0 ? 2 : 1;  // x producers (warps 6 and 7 for an even ring)
    const GemmLayout Cfg(TM, kNX);
    const int na = Cfg.na;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *xring = smem;
    uint8_t *wring = smem + kNX * Cfg.x_stage;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg.bar_off);
    uint64_t *w_full = bars, *w_empty = bars + kNW;
    uint64_t *x_full = bars + 2 * kNW, *x_empty = x_full + kNX;
    uint64_t *a_full = x_empty + kNX, *a_empty = a_full + kNAMax;
    uint64_t *d_full = a_empty + kNAMax, *d_empty = d_full + 1, *drain = d_full + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + Cfg.num_bars);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const int scale_rows = (TM + 31) / 32 * 32;
    float *xs2 = reinterpret_cast<float *>(smem + Cfg.scale_off);  // [2][scale_rows]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NT = (N + kTileN - 1) / kTileN, MT = (M + TM - 1) / TM;
    const int64_t tiles = (int64_t)NT * MT, units = tiles * splits;
    const int my_tiles = units > (int64_t)blockIdx.x ? (int)((units - 1 - blockIdx.x) / gridDim.x + 1) : 0;
    const int KW_all = K / kKW;
    // work unit i of this CTA: output tile b and K split z (weight stages
    // [wb, we)); a split writes its fp32 partial tile, summed afterwards
    struct Unit {
        int n0, m0, z, wb, we;
    };
    auto unit = [&](int i) {
        const int64_t u = (int64_t)blockIdx.x + (int64_t)i * gridDim.x;
        Unit t;
        t.z = (int)(u / tiles);
        tile_origin(u - (int64_t)t.z * tiles, NT, MT, TM, t.n0, t.m0);
        t.wb = (int)((int64_t)t.z * KW_all / splits);
        t.we = (int)((int64_t)(t.z + 1) * KW_all / splits);
        return t;
    };

    if (threadIdx.x == 0) {
        for (int i = 0; i < kNW; ++i) {
            mbar_init(&w_full[i], 1);
            mbar_init(&w_empty[i], 4);  // one arrival per dequant warp
        }
        for (int i = 0; i < kNX; ++i) {
            mbar_init(&x_full[i], 1);
            mbar_init(&x_empty[i], 1);
        }
        for (int i = 0; i < na; ++i) {
            mbar_init(&a_full[i], 4);
            mbar_init(&a_empty[i], 1);
        }
        mbar_init(d_full, 1);
        mbar_init(d_empty, 4);  // one arrival per epilogue warp
        mbar_init(drain, 1);
        *abort_flag = 0;
        mbar_fence_init();
        tma_prefetch_desc(&xmap);
        tma_prefetch_desc(&wmap);
    }
    if (warp == 1) tmem_alloc(tmem_slot, Cfg.cols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_launch_dependents();
    pdl_wait();  // x16 comes from the previous kernel
    const uint32_t tmem = *tmem_slot;
    const uint32_t d_tmem = tmem;
    const uint32_t a_tmem = tmem + Cfg.d_cols;

    if (warp == 0) {
        if (lane == 0) {
            // the weight stages of every tile, in order (g counts them)
            int g = 0;
            bool ok = true;
            for (int i = 0; ok && i < my_tiles; ++i) {
                const Unit t = unit(i);
                for (int ws = t.wb; ws < t.we; ++ws, ++g) {
                    const int wsl = g % kNW;
                    if (!mbar_wait(&w_empty[wsl], ((g / kNW) & 1) ^ 1, abort_flag, err)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&w_full[wsl], kWStageBytes);
                    tma_load_2d(wring + wsl * kWStageBytes, &wmap, ws * kWRowBytes, t.n0, &w_full[wsl]);
                }
            }
            // let every issued copy land before the CTA can exit
            for (int i = g - kNW; i < g; ++i)
                if (i >= 0) mbar_drain(&w_full[i % kNW], (i / kNW) & 1);
        }
    } else if (warp == kXProducerWarp || warp == kXProducerWarp + 1) {
        // the x stages of every tile: producer p takes stages p, p + P, ...
        const int p = warp - kXProducerWarp;
        if (lane == 0 && p < P) {
            int next = p;  // first stage (counted over all units) not issued
            int base = 0;  // x stages of the units before this one
            bool ok = true;
            for (int i = 0; ok && i < my_tiles; ++i) {
                const Unit t = unit(i);
                const int KX = (t.we - t.wb) * (kKW / kXK);
                for (int s = 0; s < KX; ++s) {
                    const int g = base + s;
                    if (g % P != p) continue;
                    const int xsl = g % kNX;
                    if (!mbar_wait(&x_empty[xsl], ((g / kNX) & 1) ^ 1, abort_flag, err)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&x_full[xsl], Cfg.x_stage);
#pragma unroll
                    for (int j = 0; j < kXChunks; ++j) {
                        const int kx = t.wb * kKW + s * kXK + 64 * j;
                        uint8_t *dst = xring + xsl * Cfg.x_stage + j * TM * 128;
                        tma_load_2d(dst, &xmap, kx, t.m0, &x_full[xsl]);
                        if (kTall)  // a TMA box is at most 256 rows: two boxes of TM / 2
                            tma_load_2d(dst + (TM / 2) * 128, &xmap, kx, t.m0 + TM / 2, &x_full[xsl]);
                    }
                    next = g + P;
                }
                base += KX;
            }
            for (int i = next - kNX; i < next; i += P)
                if (i >= 0) mbar_drain(&x_full[i % kNX], (i / kNX) & 1);
        }
    } else if (warp == 1) {
        // MMA issue; tile i waits until the epilogue has read tile i - 1
        const uint32_t idesc = idesc_f16_f32(kTileN, (uint32_t)(kTall ? 256 : TM));
        const uint32_t idesc2 = idesc_f16_f32(kTileN, (uint32_t)(kTall ? TM - 256 : 16));
        int asl = 0;
        uint32_t aph = 0;
        int base = 0;  // x stages of the units before this one
        bool ok = true;
        for (int i = 0; ok && i < my_tiles; ++i) {
            const Unit t = unit(i);
            const int KS = (t.we - t.wb) * kSlotsPerW;
            if (!__all_sync(0xffffffffu, mbar_wait(d_empty, (i & 1) ^ 1, abort_flag, err))) break;
            tc_fence_after();
            for (int s = 0; s < KS; ++s) {
#pragma unroll
                for (int u = 0; u < kXPerSlot; ++u) {
                    const int g = base + s * kXPerSlot + u;
                    ok = __all_sync(0xffffffffu, mbar_wait(&x_full[g % kNX], (g / kNX) & 1, abort_flag, err));
                    if (!ok) break;
                }
                if (!ok) break;
                if (!__all_sync(0xffffffffu, mbar_wait(&a_full[asl], aph, abort_flag, err))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < kSK / 16; ++kk) {
                        const int chunk = kk >> 2, u = chunk / kXChunks, jj = chunk % kXChunks;
                        const int g = base + s * kXPerSlot + u;
                        const uint64_t bdesc =
                            smem_desc_k128(xring + (g % kNX) * Cfg.x_stage + jj * TM * 128) + 2 * (kk & 3);
                        const uint32_t acol = a_tmem + asl * kSlotCols + kk * 8;
                        mma_f16_ts(d_tmem, acol, bdesc, idesc, (s | kk) != 0);
                        if (kTall)  // rows 256.. start 256 x 128 bytes into the chunk
                            mma_f16_ts(d_tmem + 256, acol, bdesc + (256 * 128 >> 4), idesc2, (s | kk) != 0);
                    }
#pragma unroll
                    for (int u = 0; u < kXPerSlot; ++u) mma_commit(&x_empty[(base + s * kXPerSlot + u) % kNX]);
                    mma_commit(&a_empty[asl]);
                }
                __syncwarp();
                if (++asl == na) {
                    asl = 0;
                    aph ^= 1;
                }
            }
            if (!ok) break;
            base += KS * kXPerSlot;
            if (elect_one()) mma_commit(d_full);
            __syncwarp();
        }
    } else if (warp >= 2 && warp < kXProducerWarp) {
        // warps 2..5: dequantise every tile's weight stages into the A slots
        const int quad = warp & 3;
        const int r = quad * 32 + lane;
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        int g = 0, asl = 0;
        uint32_t aph = 0;
        bool ok = true;
        for (int i = 0; ok && i < my_tiles; ++i) {
            const Unit t = unit(i);
            for (int ws = t.wb; ws < t.we && ok; ++ws, ++g) {
                const int wsl = g % kNW;
                ok = __all_sync(0xffffffffu, mbar_wait(&w_full[wsl], (g / kNW) & 1, abort_flag, err));
                if (!ok) break;
                const uint4 *row = reinterpret_cast<const uint4 *>(wring + wsl * kWStageBytes + r * kWRowBytes);
                uint32_t rw[36];
#pragma unroll
                for (int q = 0; q < 9; ++q) {
                    const uint4 v = row[q];
                    rw[4 * q + 0] = v.x;
                    rw[4 * q + 1] = v.y;
                    rw[4 * q + 2] = v.z;
                    rw[4 * q + 3] = v.w;
                }
                bool large = true;
#pragma unroll
                for (int q = 0; q < kKW / 64; ++q)
                    large = large && scale_is_large(rw[9 * q] & 0xFFFFu) && scale_is_large(rw[9 * q + 4] >> 16);
                auto stage_slots = [&](auto any_c) {
                    constexpr bool kAny = decltype(any_c)::value;
#pragma unroll
                    for (int sub = 0; sub < kSlotsPerW; ++sub) {
                        ok = __all_sync(0xffffffffu, mbar_wait(&a_empty[asl], aph ^ 1, abort_flag, err));
                        if (!ok) break;
                        tc_fence_after();
#pragma unroll
                        for (int pc = 0; pc < kChunks; ++pc) {
                            const uint32_t *wv = rw + 9 * (sub * kChunks + pc);
                            const uint32_t Q0[4] = {__funnelshift_r(wv[0], wv[1], 16),
                                                    __funnelshift_r(wv[1], wv[2], 16),
                                                    __funnelshift_r(wv[2], wv[3], 16),
                                                    __funnelshift_r(wv[3], wv[4], 16)};
                            const uint32_t Q1[4] = {wv[5], wv[6], wv[7], wv[8]};
                            uint32_t cols[32];
                            dequant_block<kAny>(wv[0] & 0xFFFFu, Q0, cols, nib_bias);
                            dequant_block<kAny>(wv[4] >> 16, Q1, cols + 16, nib_bias);
                            tmem_st32(a_tmem + lane_base + asl * kSlotCols + pc * 32, cols);
                        }
                        tmem_wait_st();
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&a_full[asl]);
                        if (++asl == na) {
                            asl = 0;
                            aph ^= 1;
                        }
                    }
                };
                if (__all_sync(0xffffffffu, large))
                    stage_slots(std::integral_constant<bool, false>{});
                else
                    stage_slots(std::integral_constant<bool, true>{});
                if (!ok) break;
                if (lane == 0) mbar_arrive(&w_empty[wsl]);
            }
        }
    } else if (warp >= kPEpiWarp0) {
        // warps 8..11: epilogue.  D[row r][column m] -> y[m][n0 + r], times
        // the x row's 2^-shift; the accumulator goes back to the MMA warp
        // once every lane's loads are done
        const int quad = warp & 3;
        const int r = quad * 32 + lane;
        const int et = threadIdx.x - kPEpiWarp0 * 32;  // 0..127
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        for (int i = 0; i < my_tiles; ++i) {
            const Unit t = unit(i);
            const int n0 = t.n0, m0 = t.m0;
            float *out = splits > 1 ? part + (size_t)t.z * M * N : nullptr;  // a split's fp32 partial tile
            // the tile's x-row scales (buffer i % 2: the other warps may
            // still read the previous tile's)
            float *xs = xs2 + (i & 1) * scale_rows;
            for (int j = et; j < scale_rows; j += 128) xs[j] = j < TM && m0 + j < M ? __ldg(xscale + m0 + j) : 0.f;
            named_bar_sync(2, 128);  // the four epilogue warps
            if (!__all_sync(0xffffffffu, mbar_wait(d_full, i & 1, abort_flag, err))) break;
            tc_fence_after();
            const int n = n0 + r;
            for (int c = 0; c < TM; c += 32) {
                uint32_t v[32];
                tmem_ld32(d_tmem + lane_base + c, v);
                float sc[32];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 t = reinterpret_cast<const float4 *>(xs + c)[q];
                    sc[4 * q] = t.x;
                    sc[4 * q + 1] = t.y;
                    sc[4 * q + 2] = t.z;
                    sc[4 * q + 3] = t.w;
                }
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int m = m0 + c + j;
                    if (c + j < TM && m < M && n < N) {
                        const float val = __uint_as_float(v[j]) * sc[j];
                        if (out)
                            out[(int64_t)m * N + n] = val;
                        else
                            store_y(y, (int64_t)m * N + n, val, ybf16 != 0);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(d_empty);
        }
    }
    __syncthreads();
    if (warp == 1) {
        if (lane == 0) {
            // every MMA issued by this CTA has finished before TMEM is released
            mma_commit(drain);
            mbar_drain(drain, 0);
        }
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, Cfg.cols);
    }
}

// ----------------------------------------------------------------- host

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

cudaError_t launch_tm(int TM, int splits, const void *x16, const float *xscale, const uint8_t *wq, float *y,
                      bool ybf16, float *part, int64_t M, int64_t N, int64_t K, cudaStream_t s, unsigned int *err) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int64_t ctas = ((N + kTileN - 1) / kTileN) * ((M + TM - 1) / TM) * splits;
    const int nx = x_ring_stages(TM, ctas, device_sm_count(dev));
    const GemmLayout Cfg(TM, nx);
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    CUtensorMap xmap, wmap;
    {
        const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
        const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
        const cuuint32_t box[2] = {64, (cuuint32_t)(TM <= 256 ? TM : TM / 2)};
        const cuuint32_t estr[2] = {1, 1};
        if (enc(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(x16), dims, strides, box,
                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
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
    // the instantiation for the tile's slot size and x ring (kNXMid and
    // kNXPair have the same depth: the slot size tells them apart)
    using Kernel = decltype(&gemm_kernel<false, kNXShort, 64, 64>);
    Kernel kernel = nullptr;
    if (slot_k(TM) == 128 && xstage_k(TM) == 128)
        kernel = TM > 256 && nx == kNXTall ? gemm_kernel<true, kNXTall, 128, 128>
                 : nx == kNXMid            ? gemm_kernel<false, kNXMid, 128, 128>
                                           : nullptr;
    else if (slot_k(TM) == 128)
        kernel = TM <= 256 && nx == kNXShort ? gemm_kernel<false, kNXShort, 128, 64> : nullptr;
    else
        kernel = nx == kNXPair    ? gemm_kernel<false, kNXPair, 64, 64>
                 : nx == kNXShort ? gemm_kernel<false, kNXShort, 64, 64>
                                  : nullptr;
    if (!kernel || (TM > 256) != (kernel == gemm_kernel<true, kNXTall, 128, 128>)) return cudaErrorInvalidConfiguration;
    const int64_t tiles = ((N + kTileN - 1) / kTileN) * ((M + TM - 1) / TM);
    const int sms = device_sm_count(dev);
    if (use_persistent(TM, nx, tiles, splits, sms)) {
        // more work units than SMs: the persistent form (one CTA per SM)
        using PK = decltype(&gemm_persistent_kernel<false, kNXShort, 128, 64>);
        const PK pk = TM > kMaxTileRowsShort ? gemm_persistent_kernel<true, kNXTall, 128, 128>
                      : nx == kNXMid         ? gemm_persistent_kernel<false, kNXMid, 128, 128>
                                             : gemm_persistent_kernel<false, kNXShort, 128, 64>;
        e = ensure_smem_attr(reinterpret_cast<const void *>(pk), (int)Cfg.smem);
        if (e != cudaSuccess) return e;
        e = launch_pdl(pk, dim3((unsigned)sms), dim3(kPThreads), Cfg.smem, s, xmap, wmap, y,
                       splits > 1 ? part : nullptr, xscale, (int)M, (int)N, (int)K, TM, splits, ybf16 ? 1 : 0, kNibbleBias,
                       err);
    } else {
        e = ensure_smem_attr(reinterpret_cast<const void *>(kernel), (int)Cfg.smem);
        if (e != cudaSuccess) return e;
        const dim3 grid((unsigned)tiles, 1, (unsigned)splits);
        e = launch_pdl(kernel, grid, dim3(kThreads), Cfg.smem, s, xmap, wmap, y, splits > 1 ? part : nullptr,
                       xscale, (int)M, (int)N, (int)K, TM, ybf16 ? 1 : 0, kNibbleBias, err);
    }
    if (e != cudaSuccess || splits == 1) return e;
    const int64_t n4 = M * N / 4;
    return launch_pdl(splitk_reduce_kernel, dim3((unsigned)((n4 + 255) / 256)), dim3(256), 0, s,
                      reinterpret_cast<const float4 *>(part), y, n4, splits, ybf16 ? 1 : 0);
}

}  // namespace

namespace {

int64_t x16_bytes(int64_t M, int64_t K) { return (M * K * 2 + 255) / 256 * 256; }
// the per-row scales of x16 (fp32), after it
int64_t xscale_bytes(int64_t M) { return (M * 4 + 255) / 256 * 256; }

// Rows of x per CTA tile.  Each extra tile dequantises every weight tile
// once more, but tiles of more than 256 rows run with a shallower x ring:
// they are used when they need at most three quarters as many tiles as
// 256-row ones (M = 272: one tile instead of two).  With `sms` known, two
// further rules look at waves of tiles (one CTA per SM):
//   * two or more 256-row tiles that leave SMs idle in a single wave: the
//     most x tiles of at least 144 rows that still fit one wave (the O and
//     down projections at M = 512: three tiles of 176 rows, 120 of 152 SMs
//     busy instead of 80);
//   * from four 256-row tiles up (M > 768), when both tilings give every SM
//     at least one tile (so K is not split): the tiling whose whole waves
//     cost less, a wave costing its tile height plus about 100 rows' worth
//     of MMA time for the tile's own work (its weight tile's
//     dequantisation, the epilogue); tall tiles are taken when that saves
//     more than 5 % (O and down at M = 2048: seven tiles of 304 rows, 280
//     tiles in two waves on 152 SMs, instead of eight of 256, 320 tiles in
//     three).
// Then the smallest multiple of 16 that covers M in that many tiles.
int tile_rows(int64_t M, int64_t N, int sms) {
    const int64_t t256 = (M + 255) / 256, tall = (M + kMaxTileRows - 1) / kMaxTileRows;
    int64_t tiles_m = 4 * tall <= 3 * t256 ? tall : t256;
    const int64_t nt = (N + kTileN - 1) / kTileN;
    if (sms > 0 && tiles_m == t256 && t256 >= 2 && t256 * nt < sms) {
        for (int64_t c = t256 + 1; c * nt <= sms && ((M + c - 1) / c + 15) / 16 * 16 >= 144; ++c) tiles_m = c;
        return (int)(((M + tiles_m - 1) / tiles_m + 15) / 16 * 16);
    }
    if (sms > 0 && t256 >= 4 && tall < t256 && tall * nt >= sms) {
        auto cost = [&](int64_t tm_count) {
            const int64_t rows = ((M + tm_count - 1) / tm_count + 15) / 16 * 16;
            return (double)((tm_count * nt + sms - 1) / sms) * (double)(rows + 100);
        };
        tiles_m = cost(tall) < 0.95 * cost(t256) ? tall : t256;
    }
    return (int)(((M + tiles_m - 1) / tiles_m + 15) / 16 * 16);
}

}  // namespace

// Split K 1..4 ways.  Score of a split = share of the SMs busy over whole
// waves (one CTA per SM) / (1 + cost of the partial tiles), the cost being
// their write and read (8 * S * M * N bytes at HBM speed) over the MMA time
// (2 * M * N * K flops at about 1 PFLOP/s): about 600 * S / K.  Each split
// keeps at least two weight stages.
int gemm_splits(int64_t M, int64_t N, int64_t K, int sms) {
    const int tm = tile_rows(M, N, sms);
    const int64_t ctas = ((N + kTileN - 1) / kTileN) * ((M + tm - 1) / tm);
    if (sms <= 0 || ctas <= 0 || (M * N) % 4 != 0) return 1;
    int best = 1;
    double best_score = 0.0;
    for (int sp = 1; sp <= 4 && K / kKW >= 2 * sp; ++sp) {
        const int64_t total = ctas * sp;
        const int64_t waves = (total + sms - 1) / sms;
        const double busy = (double)total / (double)(waves * sms);
        const double score = busy / (1.0 + (sp > 1 ? 600.0 * sp / (double)K : 0.0));
        if (score > best_score * 1.03) {
            best_score = score;
            best = sp;
        }
    }
    return best;
}

// The launch grids: all output tiles in gridDim.x, and the x pre-pass at
// one CTA per row of x.
bool gemm_shape_supported(int64_t M, int64_t N, int64_t K) {
    if (M < 1 || N < 1 || K < 1) return false;
    const int tm = tile_rows(M, N, 0);  // the most tiles any device's choice gives
    return ((N + kTileN - 1) / kTileN) * ((M + tm - 1) / tm) <= 0x7FFFFFFF && M <= 0x7FFFFFFF;
}

void gemm_plan(int64_t M, int64_t N, int64_t K, int sms, int splits, int *tile_rows_out, int *persistent_out) {
    const int tm = tile_rows(M, N, sms);
    const int64_t tiles = ((N + kTileN - 1) / kTileN) * ((M + tm - 1) / tm);
    const int nx = x_ring_stages(tm, tiles * splits, sms);
    *tile_rows_out = tm;
    *persistent_out = use_persistent(tm, nx, tiles, splits, sms) ? 1 : 0;
}

size_t gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, int splits) {
    size_t b = (size_t)x16_bytes(M, K) + (size_t)xscale_bytes(M);
    if (splits > 1) b += (size_t)splits * (size_t)M * (size_t)N * 4;
    return b;
}

cudaError_t launch_gemm(const uint16_t *x, const uint8_t *wq, float *y, bool ybf16, int64_t M, int64_t N,
                        int64_t K, void *workspace, int splits, cudaStream_t s, unsigned int *err) {
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    void *x16 = ws;
    float *xscale = reinterpret_cast<float *>(ws + x16_bytes(M, K));
    float *part = reinterpret_cast<float *>(ws + x16_bytes(M, K) + xscale_bytes(M));
    if (!gemm_shape_supported(M, N, K)) return cudaErrorInvalidValue;
    const bool long_rows = K > kXHeldShort * 8 * kXThreads && K <= kXHeldLong * 8 * kXThreads;
    cudaError_t e = launch_pdl(long_rows ? x_to_f16_kernel<kXHeldLong> : x_to_f16_kernel<kXHeldShort>, dim3((unsigned)M),
                               dim3(kXThreads), 0, s, reinterpret_cast<const uint4 *>(x),
                               reinterpret_cast<uint4 *>(x16), xscale, (int)(K / 8));
    if (e != cudaSuccess) return e;
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    return launch_tm(tile_rows(M, N, device_sm_count(dev)), splits < 1 ? 1 : splits, x16, xscale, wq, y, ybf16,
                     part, M, N, K, s, err);
}

}  // namespace q4_0
