/*
 * q4_0.h -- C ABI of libq4_0.so: matmul of bf16 activations with weights
 * stored in Q4_0, on one NVIDIA GB300 (sm_103a).
 *
 * Operation.  "Vertical disaggregation: maximizing model throughput on
 * heterogeneous silicon", section "Every cycle counts: custom kernels": the
 * CPU and the GPU paths share one Q4_0 weight format, produce deterministic
 * output, and are built from nibble unpack, dot product, scale apply, batch
 * decode and a GPU "Q4_0 -> Tensor Core" path.  This library is that GPU
 * path, written for sm_103a: a memory-bound GEMV for decode (small M) and a
 * tcgen05 tensor-core GEMM for prefill (large M), behind one dispatcher.
 *
 * Q4_0 format (the layout this library fixes; the page prints none):
 *   - a weight matrix W [N][K] is stored as N rows of K/32 blocks, row-major,
 *     one row = 18*K/32 contiguous bytes;
 *   - block = 18 bytes: bytes 0-1 an IEEE binary16 scale d (little-endian),
 *     bytes 2-17 sixteen code bytes qs[16];
 *   - element j (0..15) of the block is qs[j] & 15, element j+16 is qs[j] >> 4;
 *   - weight value w = d * (q - 8).
 *
 * Conventions for every entry point below:
 *   - Array pointers are DEVICE pointers owned by the caller unless an entry
 *     point says otherwise (q4_0_matmul_host takes host x and y; the grouped
 *     call takes host arrays of device pointers); the library keeps no
 *     pointer after the call returns and allocates nothing that outlives a
 *     call.  The one exception is the fixed scratch array of
 *     q4_0_gemm_noalloc (Q4_0_NOALLOC_SCRATCH_BYTES of device memory),
 *     which is reserved when the library is loaded on a device and held
 *     until the process exits.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Work is
 *     enqueued asynchronously on it; the caller synchronises.  Launch errors
 *     are returned; a device-side timeout is recorded in a device error word
 *     that q4_0_device_error() reads.
 *   - Arguments are validated before anything is launched; an invalid call
 *     returns a negative status and enqueues nothing.
 *   - No entry point prints or exits.  The only host-side state is
 *     process-wide caches filled once under a lock (driver entry points,
 *     per-device kernel attributes, the fixed scratch array's address);
 *     calls from several host threads are safe.
 *   - Results are deterministic: the same inputs give bit-identical outputs
 *     (fixed reduction order, no floating-point atomics).
 */
#ifndef Q4_0_H_
#define Q4_0_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define Q4_0_BLOCK_WEIGHTS 32
#define Q4_0_BLOCK_BYTES 18
#define Q4_0_VERSION 1

/* Status codes returned by every entry point. */
typedef enum {
    Q4_0_OK = 0,
    Q4_0_ERR_INVALID_ARG = -1,    /* null pointer, bad size, misaligned pointer */
    Q4_0_ERR_UNSUPPORTED = -2,    /* valid Q4_0 call outside what this build runs */
    Q4_0_ERR_CUDA = -3,           /* a CUDA runtime call or a launch failed */
    Q4_0_ERR_DEVICE_TIMEOUT = -4, /* a kernel gave up on a bounded wait */
    Q4_0_ERR_WORKSPACE = -5       /* workspace missing or too small */
} q4_0_status;

/* Library version (Q4_0_VERSION). */
int q4_0_version(void);

/* Static text for a status code; never NULL. */
const char *q4_0_status_string(int status);

/* Bytes of a Q4_0 matrix of N rows and K columns: N * K/32 * 18.
 * Returns 0 when N < 1, K < 1 or K is not a multiple of 32. */
size_t q4_0_weight_bytes(int64_t N, int64_t K);

/*
 * q4_0_quantize -- fp32 weights -> Q4_0 blocks.
 *   w   : float [N][K] row-major, device.  Values must be finite and
 *         |w| <= 8 * 65504 (the scale must fit binary16).
 *   wq  : uint8 [q4_0_weight_bytes(N, K)], device, written completely.
 *   N, K: N >= 1, K >= 32, K % 32 == 0.
 * Per block of 32 weights: d = (signed value of the max-|w| element, first
 * index on ties) / -8 in fp32; the stored scale is d rounded to binary16
 * (nearest, ties to even); each code is q = clamp(round(w / d) + 8, 0, 15)
 * with the fp32 d, IEEE division and round-half-away-from-zero; an all-zero
 * block stores d = +0 and codes 8.  Codes match the library's CPU reference
 * bit for bit.
 * Alignment: w 16 bytes; wq 2 bytes.
 * Returns Q4_0_OK, Q4_0_ERR_INVALID_ARG or Q4_0_ERR_CUDA.
 */
int q4_0_quantize(const float *w, uint8_t *wq, int64_t N, int64_t K, void *stream);

/*
 * q4_0_matmul -- y = x * W^T with W in Q4_0.
 *   x   : bf16 bit patterns [M][K] row-major, device (the __nv_bfloat16 type).
 *   wq  : Q4_0 matrix W [N][K] as above, device.
 *   y   : float [M][N] row-major, device, fully overwritten (no accumulate).
 *   M, N, K: M >= 1, N >= 1, K >= 32, K % 32 == 0 (else INVALID_ARG).
 *         K % 256 != 0 is served by copying W and x, zero-padded to K
 *         rounded up to 256, into the scratch first (one extra pass over W;
 *         the extra blocks and elements are zero, so y is unchanged).  The
 *         kernel-alone entry points below (q4_0_gemv*, q4_0_gemm*) need
 *         K % 256 == 0 and return UNSUPPORTED otherwise.
 * y[m][n] = sum_k d(n,k) * (q(n,k) - 8) * x[m][k], accumulated in fp32.
 * Dispatch: M <= 2 runs the decode GEMV on CUDA cores (exact integer dot
 * products per 32-weight block on 15-bit fixed-point x, fp32 across blocks;
 * a matrix whose per-row partial sums outgrow one launch's shared memory
 * runs as several launches over row ranges); 3 <= M <= 64, and M <= 2 with
 * K > 65536 (x no longer fits shared memory), run the batched decode on the
 * tensor cores (tiles of 16, 32 or 64 rows of x; faster than the GEMM at
 * every such M on a GB300); M > 64 runs the tcgen05 GEMM (weights dequantised to
 * binary16 tiles, x rounded to binary16, fp32 accumulation in tensor
 * memory).
 * Accuracy.  Inputs must be finite and y must stay within the fp32 range;
 * the tensor-core paths also need |w| = |d (q - 8)| <= 65504.
 * Every path accumulates in fp32 and differs from the exact sum only in the
 * form it gives w and x:
 *   - tensor-core paths (3 <= M, or M <= 2 with K > 65536): each weight
 *     rounded once to binary16 (relative error <= 2^-11); each row of x
 *     scaled by a power of two (its largest |x| to [2^14, 2^15), undone
 *     exactly at the store) and rounded to binary16: exact for every
 *     element within 2^29 of the row's largest |x|, absolute error
 *     <= 2^-39 times that largest |x| below;
 *   - integer-dot decode (M <= 2, K % 1024 == 0, K <= 65536): weights
 *     exact; x in 15-bit fixed point per 32-element block, absolute error
 *     <= 2^-14 B per element, B the largest |x| of its block;
 *   - binary16 decode (M <= 2, other K <= 65536): weights exact; x in
 *     binary16 scaled per 32-element block, absolute error <= 2^-24 B.
 * Per element, |y - y_exact| <= 1e-2 * sum_k |w x| then holds on the
 * tensor-core paths for every x whose rows span at most 2^29, on the
 * binary16 decode whenever sum_k |w| B <= 2^17 sum_k |w x|, and on the
 * integer-dot decode whenever sum_k |w| B <= 150 sum_k |w x| (with B of the
 * element's block; for N(0, 1) activations the ratio is about 3, with 1 %
 * of them 20x larger about 7).  Outside that condition the integer-dot
 * decode's error stays within 2^-14 sum_k |w| B plus fp32 rounding: one
 * element per block far above the others (a block of x spanning 2^15) with
 * its weight near zero is the case it does not cover.  The relative L2
 * error ||y - y_exact|| / ||y_exact|| is at most 2e-3 on the workloads' data
 * on every path (it is relative to ||y||, which cancellation can make
 * arbitrarily small, so it is a measured property, not a per-input bound).
 * Scratch: the tensor-core decode and GEMM (M > 64) paths need
 * q4_0_matmul_workspace_bytes(M, N, K) bytes; this entry point takes them
 * with cudaMallocAsync on `stream` and frees them with cudaFreeAsync on the
 * same stream.  Use q4_0_matmul_ws to supply the workspace yourself.
 * Alignment: x, wq and y 16 bytes.
 * Sizes this build runs (else UNSUPPORTED): M, N <= 2^30, K <= 2^24, each of
 * M*K, N*K, M*N <= 2^40; on the tensor-core decode N <= 65535 * 128 (its
 * weight tiles are a grid dimension).
 * Returns Q4_0_OK, Q4_0_ERR_INVALID_ARG, Q4_0_ERR_UNSUPPORTED or Q4_0_ERR_CUDA.
 */
int q4_0_matmul(const uint16_t *x, const uint8_t *wq, float *y,
                int64_t M, int64_t N, int64_t K, void *stream);

/* Scratch bytes q4_0_matmul needs for these sizes on the current device
 * (0 for M <= 2 when K % 256 == 0 and K <= 65536; for other K it includes
 * the zero-padded copies of W and x).  The batched-decode and GEMM parts depend on the
 * device's SM count (room for split-K partial tiles), so query on the device
 * that will run the call. */
size_t q4_0_matmul_workspace_bytes(int64_t M, int64_t N, int64_t K);

/*
 * q4_0_matmul_ws -- q4_0_matmul with caller-owned scratch.
 *   workspace       : device pointer, 256-byte aligned, at least
 *                     q4_0_matmul_workspace_bytes(M, N, K) bytes (may be
 *                     NULL when that is 0).  Contents on entry are ignored;
 *                     it is in use until the work on `stream` completes.
 *   workspace_bytes : its size.
 * Returns Q4_0_ERR_WORKSPACE when the workspace is missing or too small,
 * otherwise as q4_0_matmul.
 */
int q4_0_matmul_ws(const uint16_t *x, const uint8_t *wq, float *y,
                   int64_t M, int64_t N, int64_t K,
                   void *workspace, size_t workspace_bytes, void *stream);

/* Element types of y for q4_0_matmul_ex. */
#define Q4_0_Y_F32 0  /* float, as q4_0_matmul */
#define Q4_0_Y_BF16 1 /* bfloat16: the fp32 result rounded to nearest even */

/*
 * q4_0_matmul_ex -- q4_0_matmul with a choice of output element type: y is
 * [M][N] row-major of `y_type` (Q4_0_Y_F32 or Q4_0_Y_BF16; anything else is
 * Q4_0_ERR_INVALID_ARG), 16-byte aligned.  Every kernel accumulates in fp32
 * and rounds once at the store, so a Q4_0_Y_BF16 result equals the
 * round-to-nearest-even bfloat16 of the Q4_0_Y_F32 result of the same call.
 * Downstream layers that take bf16 activations read y directly, and the
 * store writes half the bytes.  The pages leave the output type open; this
 * is the bf16-output option of the epilogue.
 * Workspace: as q4_0_matmul_ws; workspace NULL with workspace_bytes 0 makes
 * the library take its own (cudaMallocAsync / cudaFreeAsync on `stream`).
 * Returns as q4_0_matmul_ws.
 */
int q4_0_matmul_ex(const uint16_t *x, const uint8_t *wq, void *y, int y_type,
                   int64_t M, int64_t N, int64_t K,
                   void *workspace, size_t workspace_bytes, void *stream);

/*
 * q4_0_matmul_host -- the dispatcher with x and y in host memory: one call
 * copies x ([M][K] bf16 row-major, host) into the workspace, runs the matmul
 * there, and copies y ([M][N] of `y_type`, host) back, all asynchronously on
 * `stream` in that order.  wq is the device Q4_0 matrix as for q4_0_matmul.
 * When both host buffers are page-locked memory the device can address
 * (cudaHostAlloc / cudaHostRegister; on a GB300 the Grace memory is coherent
 * with the GPU over NVLink-C2C) and 16-byte aligned there, the kernels
 * write y in host memory directly and no copy is issued: for M <= 2 a small
 * kernel first copies x into the workspace (the decode kernels read all of
 * x in every CTA), and larger M read x in host memory where they convert
 * it; either way x is read in stream order, so y of an earlier call on the
 * stream may be passed as x.  Otherwise x and y are copied with plain
 * cudaMemcpyAsync (page-locked
 * buffers let the copies overlap the host).  Either way the caller
 * synchronises `stream` before reading y (or reusing x).
 * Workspace: device memory, 16-byte aligned, of at least
 * q4_0_matmul_host_workspace_bytes(M, N, K, y_type) bytes: the device copies
 * of x and y (each rounded up to 256 bytes) and the matmul's own scratch;
 * a missing, misaligned or small workspace is Q4_0_ERR_WORKSPACE.
 * The size query returns 0 for arguments the call would reject.
 * Returns as q4_0_matmul_ex; a failed copy is Q4_0_ERR_CUDA.
 */
size_t q4_0_matmul_host_workspace_bytes(int64_t M, int64_t N, int64_t K, int y_type);
int q4_0_matmul_host(const uint16_t *x_host, const uint8_t *wq, void *y_host, int y_type,
                     int64_t M, int64_t N, int64_t K,
                     void *workspace, size_t workspace_bytes, void *stream);

/*
 * q4_0_matmul_grouped -- G independent problems y_g = x_g * W_g^T that share
 * M, issued together on `stream`:
 *   G        : 0 .. 4096 problems (0 does nothing).
 *   x, wq, y : host arrays of G device pointers; x_g bf16 [M][K_g], wq_g
 *              Q4_0 [N_g][K_g], y_g [M][N_g] of `y_type` (Q4_0_Y_F32 or
 *              Q4_0_Y_BF16), each as in q4_0_matmul_ex.  The arrays are
 *              read during the call only.
 *   N, K     : host arrays of the G sizes.
 * With M == 1 and K_g % 1024 == 0 (K_g <= 65536), consecutive problems run
 * as one persistent decode launch per group of up to eight (as many as one
 * SM's shared memory holds): every CTA streams its share of each problem's
 * weights back to back, so the launch front and tail are paid once per group
 * rather than once per matrix.  Any other problem runs as q4_0_matmul_ex
 * with library-allocated scratch (cudaMallocAsync on `stream`), in order.
 * Each y_g equals the q4_0_matmul_ex result of its problem bit for bit.
 * Every problem is checked before anything is launched.  The problems must
 * not overlap in y with each other or with any x or W.
 * Returns Q4_0_OK, Q4_0_ERR_INVALID_ARG, Q4_0_ERR_UNSUPPORTED or Q4_0_ERR_CUDA.
 */
int q4_0_matmul_grouped(int G, const uint16_t *const *x, const uint8_t *const *wq, void *const *y, int y_type,
                        int64_t M, const int64_t *N, const int64_t *K, void *stream);

/* Kernel launches a q4_0_matmul_grouped call with these sizes makes on the
 * current device when the grouped decode takes every problem; -1 when it
 * does not take them all (or there is no device). */
int q4_0_matmul_grouped_launches(int G, int64_t M, const int64_t *N, const int64_t *K);

/*
 * q4_0_gemv -- the decode kernels alone (what q4_0_matmul runs for
 * M <= 64).  Same arguments, layout and result contract as q4_0_matmul;
 * M <= 64 (larger M is UNSUPPORTED).  M <= 2 with K <= 65536 needs no
 * scratch; on the tensor-core decode (3 <= M <= 64, or larger K) x is first
 * rounded to binary16 tensor-core tiles, and when K is split across CTAs
 * their partial tiles and counters sit beside them:
 * q4_0_gemv_workspace_bytes(M, K) bytes of scratch, which this entry point
 * takes with cudaMallocAsync / cudaFreeAsync on `stream`.
 */
int q4_0_gemv(const uint16_t *x, const uint8_t *wq, float *y,
              int64_t M, int64_t N, int64_t K, void *stream);

/* Scratch bytes of the decode kernels on the current device (0 for M > 64,
 * and for M <= 2 with K <= 65536): the binary16 x tiles plus room for two
 * split-K partial tiles (and counters) per SM, whatever N is. */
size_t q4_0_gemv_workspace_bytes(int64_t M, int64_t K);

/*
 * q4_0_gemv_ws -- q4_0_gemv with caller-owned scratch: workspace 256-byte
 * aligned, at least q4_0_gemv_workspace_bytes(M, K) bytes (may be NULL when
 * that is 0), in use until the work on `stream` completes.  Returns
 * Q4_0_ERR_WORKSPACE when it is missing, misaligned or too small, otherwise
 * as q4_0_gemv.
 */
int q4_0_gemv_ws(const uint16_t *x, const uint8_t *wq, float *y,
                 int64_t M, int64_t N, int64_t K,
                 void *workspace, size_t workspace_bytes, void *stream);

/*
 * q4_0_gemm -- the tcgen05 prefill kernel alone (what q4_0_matmul runs for
 * M > 64), usable at any M >= 1 for cross-checks.  Workspace as in
 * q4_0_matmul_ws: q4_0_gemm_workspace_bytes(M, N, K) bytes on the current
 * device -- x rounded to binary16 and, when the output tiles alone would
 * leave SMs idle, fp32 partial tiles of a 2- to 4-way split of K (summed
 * afterwards in split order, so results stay deterministic).  A workspace
 * large enough for x alone runs without the split.
 */
size_t q4_0_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K);
int q4_0_gemm(const uint16_t *x, const uint8_t *wq, float *y,
              int64_t M, int64_t N, int64_t K,
              void *workspace, size_t workspace_bytes, void *stream);

/*
 * q4_0_gemm_plan -- the launch q4_0_gemm makes for (M, N, K) with its
 * default workspace (q4_0_gemm_workspace_bytes) on the current device, and
 * that q4_0_matmul makes for M > 64.  No work is launched.
 *   *tile_rows  : x rows per output tile (a multiple of 16, at most 320)
 *   *splits     : ways K is split over CTAs (1..4; the fp32 partial tiles
 *                 are summed in split order by a second kernel afterwards)
 *   *persistent : 1 when one CTA per SM takes several work units (output
 *                 tiles, or tile x K-split units) in turn -- tiles of more
 *                 than 128 rows, more units than SMs -- else 0 (one CTA per
 *                 tile and split)
 * Errors: Q4_0_ERR_INVALID_ARG for a null output pointer, M, N < 1 or
 * K % 256 != 0; Q4_0_ERR_CUDA when no device is current.
 */
int q4_0_gemm_plan(int64_t M, int64_t N, int64_t K, int *tile_rows, int *splits, int *persistent);

/*
 * q4_0_gemm_noalloc -- q4_0_gemm for callers that cannot allocate device
 * memory and have no workspace to hand over.  The paper has no counterpart:
 * this entry point exists for callers where the CUDA allocator must not be
 * entered (host callbacks, real-time loops with no allocation after
 * start-up, plug-ins whose host owns every device byte).
 *   x, wq, y, M, N, K, stream : as in q4_0_gemm, and the same kernels run,
 *   with one difference: this entry point never splits K over several CTAs
 *   (the array holds the binary16 copy of x only).  q4_0_gemm splits K when
 *   the output tiles alone leave SMs idle, and a split sums in another
 *   order, so the two results can differ in the last bits (both meet the
 *   result contract of q4_0_matmul), and for few output tiles this entry
 *   point keeps fewer SMs busy.
 * Scratch: a fixed array of Q4_0_NOALLOC_SCRATCH_BYTES in device memory,
 * reserved when the library is loaded on a GPU and held until the process
 * exits; nothing is allocated or freed per call.  It fits M * K * 2 bytes,
 * i.e. M * K <= 16 Mi elements; larger calls return Q4_0_ERR_WORKSPACE and
 * launch nothing.
 * The array is shared by every call on a device: calls whose kernels overlap
 * on the GPU (unordered streams) race on it -- order them on one stream.
 * The first call on each device looks up the array's address; make it before
 * any stream capture begins.
 * Returns Q4_0_OK, Q4_0_ERR_INVALID_ARG, Q4_0_ERR_UNSUPPORTED,
 * Q4_0_ERR_WORKSPACE or Q4_0_ERR_CUDA.
 */
#define Q4_0_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
int q4_0_gemm_noalloc(const uint16_t *x, const uint8_t *wq, float *y,
                      int64_t M, int64_t N, int64_t K, void *stream);

/*
 * q4_0_device_error -- read and clear the device error word of the current
 * device.  Synchronises the device.  *code receives Q4_0_OK or
 * Q4_0_ERR_DEVICE_TIMEOUT (a kernel gave up on a bounded wait and left its
 * output incomplete).  Returns Q4_0_OK or Q4_0_ERR_CUDA.
 */
int q4_0_device_error(int *code);

/*
 * q4_0_selftest_wait_timeout -- exercise the failure path of the bounded
 * waits.  Launches one thread that waits on an mbarrier nothing arrives on,
 * gives up after `limit_us` microseconds (1 .. 1e6), records
 * Q4_0_ERR_DEVICE_TIMEOUT in the device error word and returns; it traps
 * nothing and leaves the context usable.  Every pipeline wait of the matmul
 * kernels fails the same way (after about two seconds).  Read the result with
 * q4_0_device_error().
 * Returns Q4_0_OK, Q4_0_ERR_INVALID_ARG or Q4_0_ERR_CUDA.
 */
int q4_0_selftest_wait_timeout(int64_t limit_us, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* Q4_0_H_ */
