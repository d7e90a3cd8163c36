"""Q4_0 matmul on the device against the oracle (all through the C ABI)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_common import check_full, check_sampled, lib, wq_dev, x_dev
from q4_weight_only_gb300 import synth

pytestmark = pytest.mark.gpu


# q4_0_matmul sends M up to this to the decode kernels, larger M to the GEMM
DECODE_MAX_M = 64


def case(seed, M, N, K, outlier_blocks=0.0, act_outliers=0.0):
    w, x = synth.small_case(seed, M, N, K, outlier_block_frac=outlier_blocks,
                            act_outlier_frac=act_outliers)
    return x, oracle.get().quantize(w)


# ------------------------------------------------------------ small, full

SMALL_GEMV = [(1, 1, 256), (1, 2, 256), (1, 3, 512), (1, 200, 1280), (1, 257, 2304),
              (2, 129, 1024), (3, 64, 768), (4, 300, 2048), (5, 77, 4352), (8, 1000, 1280),
              (13, 33, 2560), (16, 512, 1024), (31, 65, 1536), (32, 256, 3072),
              # K % 1024 == 0 with M <= 2: the integer-dot decode kernel
              (1, 1, 1024), (1, 3, 2048), (1, 31, 3072), (2, 200, 1024), (2, 257, 4096),
              (1, 1000, 7168), (2, 5, 17408), (1, 4099, 5120),
              # 33 <= M <= 64: the tensor-core decode's 64-row tile (x stages of 128 k)
              (33, 100, 1024), (40, 1000, 5120), (48, 300, 2048), (64, 129, 1536), (64, 5120, 17408)]


@pytest.mark.parametrize("M,N,K", SMALL_GEMV)
def test_gemv_small(M, N, K):
    q4 = lib()
    x, wq = case(1000 + M * 7 + N, M, N, K, outlier_blocks=0.05, act_outliers=0.01)
    check_full(q4.gemv(x_dev(x), wq_dev(wq), N, K), x, wq, N, K)


SMALL_GEMM = [(1, 128, 256), (16, 128, 256), (17, 200, 512), (32, 384, 768), (33, 128, 256),
              (64, 1000, 1280), (65, 129, 2304), (100, 256, 1024), (128, 640, 512),
              (129, 300, 768), (256, 128, 1024), (300, 520, 1536), (513, 384, 512),
              # one x tile of more than 256 rows: a second MMA per k step
              (257, 130, 512), (272, 384, 1024), (320, 256, 2048), (321, 200, 512)]


@pytest.mark.parametrize("M,N,K", SMALL_GEMM)
def test_gemm_small(M, N, K):
    q4 = lib()
    x, wq = case(2000 + M * 7 + N, M, N, K, outlier_blocks=0.05)
    check_full(q4.gemm(x_dev(x), wq_dev(wq), N, K), x, wq, N, K)


def test_dispatch_matches_kernels_bitwise():
    q4 = lib()
    for M in (1, 7, 32, 33, 64, 65, 200):
        x, wq = case(3000 + M, M, 384, 1024)
        xd, wd = x_dev(x), wq_dev(wq)
        y = q4.matmul(xd, wd, 384, 1024)
        ref = q4.gemv(xd, wd, 384, 1024) if M <= DECODE_MAX_M else q4.gemm(xd, wd, 384, 1024)
        assert torch.equal(y, ref)
        assert torch.equal(q4.matmul_alloc(xd, wd, 384, 1024), y)


def test_gemm_split_k_matches_unsplit():
    """A workspace with room only for x (binary16, and the rows' scales) runs
    the GEMM unsplit; the default workspace may split K (few output tiles).
    Both meet the tolerance."""
    q4 = lib()
    M, N, K = 272, 384, 5120                       # 3 x 2 output tiles: K gets split
    x, wq = case(8100, M, N, K)
    xd, wd = x_dev(x), wq_dev(wq)
    split = q4.gemm(xd, wd, N, K)
    ws_x_only = torch.empty(q4.lib().q4_0_gemm_workspace_bytes(M, N, K), dtype=torch.uint8, device="cuda")
    small = ws_x_only[: (M * K * 2 + 255) // 256 * 256 + (M * 4 + 255) // 256 * 256]
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    st = q4.lib().q4_0_gemm(xd.data_ptr(), wd.data_ptr(), y.data_ptr(), M, N, K, small.data_ptr(),
                            small.numel(), None)
    assert st == q4.OK
    check_full(split, x, wq, N, K)
    check_full(y, x, wq, N, K)
    assert q4.lib().q4_0_gemm_workspace_bytes(M, N, K) > small.numel()


def test_large_scales_take_the_exact_fallback():
    """Blocks whose scale d reaches |d| >= 64 (|w| up to ~1000) dequantise
    through the exponent-bias route; mixed with ordinary blocks in one
    matrix, through the batched decode and the GEMM."""
    q4 = lib()
    g = synth.generator(8200)
    N, K = 300, 2048
    w = synth.weights(g, N, K)
    big = g.random((N, K // 32)) < 0.1
    w.reshape(N, K // 32, 32)[big] *= np.float32(30000.0)     # |d| around 100..300
    wq = oracle.get().quantize(w)
    codes, dbits = oracle.get().unpack(wq, N, K)
    assert ((dbits & 0x7FFF) >= 0x5400).any() and ((dbits & 0x7FFF) < 0x5400).any()
    for M in (4, 20, 64):
        x = synth.to_bf16_bits(synth.activations_f32(g, M, K))
        check_full(q4.matmul(x_dev(x), wq_dev(wq), N, K), x, wq, N, K)


def test_small_scales_take_the_shift_route():
    """Every block with |d| < 2^-10 (normal, subnormal and zero scales): the
    tensor-core dequantisation cannot use d / 16 there and shifts the high
    nibbles instead.  All blocks are small, so an error in that route is not
    hidden by larger blocks in the error budget."""
    q4 = lib()
    g = synth.generator(8300)
    N, K = 300, 2048
    w = synth.weights(g, N, K) * np.float32(0.03)                  # |d| around 2^-12
    blocks = w.reshape(N, K // 32, 32)
    sub = g.random((N, K // 32)) < 0.2
    blocks[sub] *= np.float32(1e-3)                                # subnormal binary16 scales
    blocks[g.random((N, K // 32)) < 0.05] = 0.0                    # d = +0
    wq = oracle.get().quantize(w)
    codes, dbits = oracle.get().unpack(wq, N, K)
    assert ((dbits & 0x7C00) < 0x1400).all()
    assert ((dbits & 0x7C00) == 0).any() and ((dbits & 0x7FFF) != 0).any() and (dbits == 0).any()
    for M in (4, 20, 64):
        x = synth.to_bf16_bits(synth.activations_f32(g, M, K))
        check_full(q4.matmul(x_dev(x), wq_dev(wq), N, K), x, wq, N, K)


def test_gemv_and_gemm_agree():
    q4 = lib()
    for M in (1, 16, 32):
        x, wq = case(4000 + M, M, 512, 2048, act_outliers=0.01)
        xd, wd = x_dev(x), wq_dev(wq)
        a = q4.gemv(xd, wd, 512, 2048).double().cpu().numpy()
        b = q4.gemm(xd, wd, 512, 2048).double().cpu().numpy()
        _, absum = oracle.get().matmul(x, wq, 512, 2048)
        assert oracle.check(a, b, absum)["ok"]


def test_deterministic():
    q4 = lib()
    for M, N, K in ((1, 5000, 5120), (8, 700, 2048), (300, 500, 1024)):
        x, wq = case(5000 + M, M, N, K)
        xd, wd = x_dev(x), wq_dev(wq)
        y1 = q4.matmul(xd, wd, N, K).clone()
        y2 = q4.matmul(xd, wd, N, K)
        assert torch.equal(y1, y2)


def test_batched_split_k_repeats_bitwise():
    """Batched decode of the down projection (K = 17408) splits K seven ways
    per 128-row tile: the splits write partial tiles to the workspace and the
    last one to count in sums them in split order.  Repeats of the same call
    must agree bit for bit: a partial read before it is complete, a stale
    weight stage or a counter left over from the previous call shows up here
    as differing outputs."""
    q4 = lib()
    N, K = synth.SHAPES["down"]
    wd = wq_dev(oracle.get().quantize(synth.decode_weights("down")))
    for M in (16, 32):
        xd = x_dev(synth.batched_x("down", M))
        y0 = q4.matmul(xd, wd, N, K).clone()
        for _ in range(12):
            assert torch.equal(q4.matmul(xd, wd, N, K), y0)
        assert q4.device_error() == 0


def test_batched_split_k_any_workspace_contents():
    """The split-K tile counters live in caller scratch that is never
    cleared: a counter carries the token of the launch that claimed it, and
    anything else counts as zero.  Workspaces filled with zeros, all-ones or
    random bytes give the same result bit for bit, and so does a workspace
    reused after calls of other shapes."""
    q4 = lib()
    N, K = synth.SHAPES["o"]
    wd = wq_dev(oracle.get().quantize(synth.decode_weights("o")))
    for M in (4, 16, 32):
        xd = x_dev(synth.batched_x("o", M))
        nbytes = int(q4.lib().q4_0_matmul_workspace_bytes(M, N, K))
        ref = q4.matmul(xd, wd, N, K, workspace=torch.zeros(nbytes, dtype=torch.uint8, device="cuda")).clone()
        g = torch.Generator(device="cuda").manual_seed(M)
        fills = (torch.full((nbytes,), 0xFF, dtype=torch.uint8, device="cuda"),
                 torch.randint(0, 256, (nbytes,), dtype=torch.uint8, device="cuda", generator=g))
        for ws in fills:
            assert torch.equal(q4.matmul(xd, wd, N, K, workspace=ws), ref)
            assert torch.equal(q4.matmul(xd, wd, N, K, workspace=ws), ref)
        # the same scratch through calls of other shapes in between
        ws = fills[1]
        x2, w2 = case(8100 + M, M, 700, 2048)
        q4.matmul(x_dev(x2), wq_dev(w2), 700, 2048, workspace=ws)
        assert torch.equal(q4.matmul(xd, wd, N, K, workspace=ws), ref)
        assert q4.device_error() == 0


def test_output_guards_untouched():
    q4 = lib()
    for M, N, K in ((1, 33, 256), (5, 130, 512), (70, 130, 512)):
        x, wq = case(6000 + M, M, N, K)
        pad = 64
        buf = torch.full((M * N + 2 * pad,), float("nan"), device="cuda")
        out = buf[pad:pad + M * N].view(M, N)
        q4.matmul(x_dev(x), wq_dev(wq), N, K, out=out)
        assert torch.isnan(buf[:pad]).all() and torch.isnan(buf[pad + M * N:]).all()
        check_full(out, x, wq, N, K)


def test_device_argument_errors():
    q4 = lib()
    x, wq = case(7000, 40, 128, 256)
    xd, wd = x_dev(x), wq_dev(wq)
    y = torch.empty((40, 128), dtype=torch.float32, device="cuda")
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    st = q4.lib().q4_0_gemm(xd.data_ptr(), wd.data_ptr(), y.data_ptr(), 40, 128, 256,
                            small.data_ptr(), small.numel(), None)
    assert st == q4.ERR_WORKSPACE
    st = q4.lib().q4_0_matmul_ws(xd.data_ptr(), wd.data_ptr(), y.data_ptr(), 40, 128, 256,
                                 None, 0, None)
    assert st == q4.ERR_WORKSPACE
    big = torch.empty(2 * 40 * 256 + 8, dtype=torch.bfloat16, device="cuda")
    shifted = big[1:1 + 40 * 256].view(40, 256)       # 2-byte aligned only
    shifted.copy_(xd)
    with pytest.raises(q4.Q4Error) as e:
        q4.matmul(shifted, wd, 128, 256)
    assert e.value.status == q4.ERR_INVALID_ARG
    assert q4.device_error() == 0


def test_gemv_scratch_paths_agree():
    """q4_0_gemv (library-allocated scratch) and q4_0_gemv_ws (caller's
    workspace, here with slack) give identical bits; a workspace one byte
    short is refused before anything is launched."""
    q4 = lib()
    for M in (1, 3, 16, 17, 32, 33, 64):
        x, wq = case(7100 + M, M, 300, 1536)
        xd, wd = x_dev(x), wq_dev(wq)
        a = q4.gemv(xd, wd, 300, 1536)
        need = q4.lib().q4_0_gemv_workspace_bytes(M, 1536)
        ws = torch.empty(need + 4096, dtype=torch.uint8, device="cuda")
        b = q4.gemv(xd, wd, 300, 1536, workspace=ws)
        c = q4.gemv_alloc(xd, wd, 300, 1536)
        torch.cuda.synchronize()
        assert torch.equal(a, b) and torch.equal(a, c)
        if need:
            y = torch.empty((M, 300), dtype=torch.float32, device="cuda")
            st = q4.lib().q4_0_gemv_ws(xd.data_ptr(), wd.data_ptr(), y.data_ptr(), M, 300, 1536,
                                       ws.data_ptr(), need - 1, None)
            assert st == q4.ERR_WORKSPACE
    assert q4.device_error() == 0


GENERAL_K = [(1, 300, 32), (1, 257, 96), (2, 100, 288), (1, 1000, 5152),   # decode kernels
             (3, 64, 160), (16, 300, 1056), (32, 129, 2080),                   # tensor-core decode
             (64, 300, 800), (300, 520, 1312)]                                 # GEMM


@pytest.mark.parametrize("M,N,K", GENERAL_K)
def test_general_k(M, N, K):
    """K % 32 == 0 but not a multiple of 256: the dispatcher copies W and x,
    zero-padded, into its scratch and runs the padded problem; results meet
    the oracle tolerance and the allocating path gives the same bits."""
    q4 = lib()
    x, wq = case(9300 + M * 3 + K, M, N, K, outlier_blocks=0.05, act_outliers=0.01)
    xd, wd = x_dev(x), wq_dev(wq)
    y = q4.matmul(xd, wd, N, K)
    check_full(y, x, wq, N, K)
    assert torch.equal(q4.matmul_alloc(xd, wd, N, K), y)
    assert q4.device_error() == 0


BF16_OUT = [(1, 300, 2048),        # integer-dot decode
            (1, 200, 1280),        # general-K decode
            (2, 129, 1024),        # integer-dot decode, two rows
            (3, 300, 1536), (16, 512, 1024), (32, 256, 3072),   # tensor-core decode
            (64, 1000, 1280),      # GEMM
            (272, 384, 5120)]      # GEMM with a K split and the partial-tile sum


@pytest.mark.parametrize("M,N,K", BF16_OUT)
def test_bf16_output_is_the_rounded_f32_output(M, N, K):
    """q4_0_matmul_ex with bf16 y: every path rounds its fp32 result once
    (nearest even) at the store, so the bits equal bf16(fp32 y) of the same
    call, with the caller's workspace and with library-allocated scratch; and
    the result meets the oracle tolerance."""
    q4 = lib()
    x, wq = case(9100 + M, M, N, K, outlier_blocks=0.05, act_outliers=0.01)
    xd, wd = x_dev(x), wq_dev(wq)
    y32 = q4.matmul(xd, wd, N, K)
    y16 = q4.matmul(xd, wd, N, K, out_dtype=torch.bfloat16)
    assert y16.dtype == torch.bfloat16
    assert torch.equal(y16.view(torch.int16), y32.to(torch.bfloat16).view(torch.int16))
    alloc = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    st = q4.lib().q4_0_matmul_ex(xd.data_ptr(), wd.data_ptr(), alloc.data_ptr(), q4.Y_BF16, M, N, K,
                                 None, 0, None)
    assert st == q4.OK
    assert torch.equal(alloc.view(torch.int16), y16.view(torch.int16))
    check_full(y16.float(), x, wq, N, K)
    assert q4.device_error() == 0


# --------------------------------------------------------- workload sizes

def test_pr1():
    q4 = lib()
    w, x = synth.pr1()
    wq = oracle.get().quantize(w)
    check_full(q4.matmul(x_dev(x), wq_dev(wq), 256, 1024), x, wq, 256, 1024)


@pytest.mark.parametrize("shape", synth.SHAPE_ORDER)
def test_decode_full(shape):
    q4 = lib()
    N, K = synth.SHAPES[shape]
    w, x = synth.decode(shape)
    wq = oracle.get().quantize(w)
    check_full(q4.matmul(x_dev(x), wq_dev(wq), N, K), x, wq, N, K)


@pytest.mark.parametrize("shape", synth.SHAPE_ORDER)
def test_batched(shape):
    q4 = lib()
    N, K = synth.SHAPES[shape]
    wq = oracle.get().quantize(synth.decode_weights(shape))
    wd = wq_dev(wq)
    for M in synth.BATCHED_M:
        x = synth.batched_x(shape, M)
        y = q4.matmul(x_dev(x), wd, N, K)
        if M == 4 and shape in ("o", "qkv"):
            check_full(y, x, wq, N, K)
        else:
            check_sampled(y, x, wq, N, K, seed=M)


@pytest.mark.parametrize("shape", synth.SHAPE_ORDER)
def test_prefill(shape):
    q4 = lib()
    N, K = synth.SHAPES[shape]
    wq = oracle.get().quantize(synth.prefill_weights(shape))
    wd = wq_dev(wq)
    for M in synth.PREFILL_M:
        x = synth.prefill_x(shape, M)
        y = q4.matmul(x_dev(x), wd, N, K)
        check_sampled(y, x, wq, N, K, seed=M)
        del y
        torch.cuda.empty_cache()
    assert q4.device_error() == 0


@pytest.mark.parametrize("shape", ["qkv", "down"])
def test_chunked_prefill_m272(shape):
    """A 256-token prefill chunk and a 16-row decode batch as one M = 272 call."""
    q4 = lib()
    N, K = synth.SHAPES[shape]
    wq = oracle.get().quantize(synth.prefill_weights(shape))
    w, x = synth.small_case(500 + synth.SHAPE_ORDER.index(shape), 272, 8, K, act_outlier_frac=0.01)
    y = q4.matmul(x_dev(x), wq_dev(wq), N, K)
    check_sampled(y, x, wq, N, K, seed=272)


def test_matmul_host_equals_device_call():
    """q4_0_matmul_host gives bit for bit what the device-buffer dispatcher
    gives: with page-locked buffers (read and written by the kernels in
    place) and with pageable ones (copied in and out)."""
    q4 = lib()
    # M <= 2: x staged into the workspace by a copy kernel; 3 <= M <= 64: the
    # batched decode's pre-pass reads host x before its dependency wait
    # (K = 9216 and 17408: rows staged in shared memory by bulk copies)
    for M, N, K in ((1, 1000, 5120), (2, 300, 1024), (16, 300, 2048), (64, 260, 1024), (300, 200, 512),
                    (1, 100, 96), (3, 200, 9216), (16, 256, 17408)):
        x, wq = case(8400 + M, M, N, K)
        wd = wq_dev(wq)
        x_pageable = torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16)
        for pinned in (True, False):
            xh = x_pageable.pin_memory() if pinned else x_pageable
            for dt in (torch.float32, torch.bfloat16):
                ref = q4.matmul(xh.cuda(), wd, N, K, out_dtype=dt).cpu()
                out = torch.empty((M, N), dtype=dt, pin_memory=pinned)
                st = torch.cuda.current_stream()
                y = q4.matmul_host(xh, wd, N, K, out=out, out_dtype=dt, stream=st)
                st.synchronize()
                assert not y.is_cuda and y.dtype == dt
                assert torch.equal(y, ref), (M, N, K, dt, pinned)


def test_matmul_host_chained_through_host_memory():
    """y of one q4_0_matmul_host call (bf16, page-locked) passed as x of the
    next on the same stream, with no synchronisation between them: the second
    call reads x in stream order, so both match the same chain on device
    buffers bit for bit (M = 1 copies x into the workspace first; M = 16
    reads it in its x pre-pass)."""
    q4 = lib()
    K0, N0, N1 = 1024, 1024, 512
    for M in (1, 16):
        x, wq0 = case(8500 + M, M, N0, K0)
        _, wq1 = case(8600 + M, M, N1, N0)
        wd0, wd1 = wq_dev(wq0), wq_dev(wq1)
        xh = torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).pin_memory()
        st = torch.cuda.current_stream()
        for rep in range(3):
            y0 = torch.full((M, N0), float("nan"), dtype=torch.bfloat16, pin_memory=True)
            y1 = torch.empty((M, N1), dtype=torch.float32, pin_memory=True)
            q4.matmul_host(xh, wd0, N0, K0, out=y0, out_dtype=torch.bfloat16, stream=st)
            q4.matmul_host(y0, wd1, N1, N0, out=y1, stream=st)
            st.synchronize()
            r0 = q4.matmul(xh.cuda(), wd0, N0, K0, out_dtype=torch.bfloat16)
            r1 = q4.matmul(r0, wd1, N1, N0).cpu()
            assert torch.equal(y0, r0.cpu()), (M, rep)
            assert torch.equal(y1, r1), (M, rep)


def test_graph_capture_replays_bitwise():
    """A decode step captured into a CUDA graph (decode, batched decode and
    GEMM calls back to back under programmatic dependent launch, each with
    its own workspace) replays to the same bits as the direct calls, and
    every replayed output meets the oracle tolerance."""
    q4 = lib()
    calls, host = [], []
    for M, N, K in ((1, 1000, 5120), (2, 300, 1024), (16, 520, 2048), (40, 300, 1024), (272, 260, 1024),
                    (1, 100, 96)):
        x, wq = case(8600 + M + N, M, N, K)
        xd, wd = x_dev(x), wq_dev(wq)
        ws = torch.empty(max(1, q4.lib().q4_0_matmul_workspace_bytes(M, N, K)), dtype=torch.uint8, device="cuda")
        y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        calls.append((xd, wd, N, K, ws, y))
        host.append((x, wq, N, K))
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        ref = [q4.matmul(xd, wd, N, K, workspace=ws, stream=st).clone() for xd, wd, N, K, ws, _ in calls]
        st.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            for xd, wd, N, K, ws, y in calls:
                q4.matmul(xd, wd, N, K, out=y, workspace=ws, stream=st)
        for _ in range(3):
            for *_, y in calls:
                y.fill_(float("nan"))
            g.replay()
            st.synchronize()
            for r, (*_, y) in zip(ref, calls):
                assert torch.equal(y, r)
    for (x, wq, N, K), (*_, y) in zip(host, calls):
        check_full(y, x, wq, N, K)
    assert q4.device_error() == 0


def test_concurrent_streams():
    """Calls on two streams at once (each with its own workspace and output)
    give the results of the same calls run alone."""
    q4 = lib()
    jobs = []
    for i, (M, N, K) in enumerate(((1, 3000, 5120), (16, 1500, 2048), (300, 700, 1024))):
        x, wq = case(8700 + i, M, N, K)
        xd, wd = x_dev(x), wq_dev(wq)
        ref = q4.matmul(xd, wd, N, K)
        jobs.append((xd, wd, N, K, ref))
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    for rep in range(4):
        for j, (xd, wd, N, K, ref) in enumerate(jobs):
            st = streams[(rep + j) % 2]
            with torch.cuda.stream(st):
                outs.append((q4.matmul(xd, wd, N, K, stream=st), ref))
    torch.cuda.synchronize()
    for y, ref in outs:
        assert torch.equal(y, ref)
    assert q4.device_error() == 0


def test_prefill_down_m512_every_output():
    """The down projection (K = 17408: 68 weight stages per tile, the longest
    k loop of the configurations) at M = 512, every output against the
    oracle rather than a sample."""
    q4 = lib()
    N, K = synth.SHAPES["down"]
    wq = oracle.get().quantize(synth.prefill_weights("down"))
    x = synth.prefill_x("down", 512)
    y = q4.matmul(x_dev(x), wq_dev(wq), N, K)
    check_full(y, x, wq, N, K)
    assert q4.device_error() == 0


@pytest.mark.parametrize("M,K", [(256, 1024), (128, 512)])
def test_gemm_whole_waves_and_a_ragged_wave(M, K):
    """More output tiles than CTA slots, the last wave only partly full:
    256-row tiles give one slot per SM, 128-row tiles two (paired CTAs with
    the shallow x ring).  Every output against the oracle, and the result
    repeats bit for bit."""
    q4 = lib()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    slots = sms * (2 if M <= 128 else 1)
    N = 128 * (slots + 20)                      # one whole wave, then 20 tiles
    x, wq = case(9500 + M, M, N, K, outlier_blocks=0.05, act_outliers=0.01)
    xd, wd = x_dev(x), wq_dev(wq)
    y = q4.gemm(xd, wd, N, K)
    check_full(y, x, wq, N, K)
    assert torch.equal(q4.gemm(xd, wd, N, K), y)
    assert q4.device_error() == 0


def test_gemm_plan():
    """The launch plan the library reports for the prefill shapes at M =
    2048: QKV and gate+up in 256-row tiles, O and down (40 weight tiles) in
    seven tall tiles of 304 rows -- 280 tiles, two waves on 152 SMs, instead
    of 320 in three -- all persistent and unsplit; M = 272 is one tall
    tile, persistent for gate+up (more tiles than SMs); small M runs one CTA
    per tile."""
    q4 = lib()
    p = q4.gemm_plan(2048, 7168, 5120)
    assert p == {"tile_rows": 256, "splits": 1, "persistent": True}
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        for K in (5120, 17408):
            p = q4.gemm_plan(2048, 5120, K)
            assert p == {"tile_rows": 304, "splits": 1, "persistent": True}, p
            # M = 512: two 256-row tiles leave SMs idle in one wave; three of
            # 176 rows fill 120 of 152
            p = q4.gemm_plan(512, 5120, K)
            assert p == {"tile_rows": 176, "splits": 1, "persistent": False}, p
    p = q4.gemm_plan(272, 34816, 5120)
    assert p == {"tile_rows": 272, "splits": 1, "persistent": True}
    assert not q4.gemm_plan(96, 5120, 5120)["persistent"]
    with pytest.raises(q4.Q4Error):
        q4.gemm_plan(64, 128, 300)


def test_gemm_wave_aware_tall_tiles_every_output():
    """M = 2048 against 40 weight tiles takes seven tall x tiles (six of
    304 rows and a ragged one of 224) in the persistent form: every output
    against the oracle, bitwise repeatable, and equal to the same call made
    through q4_0_matmul."""
    q4 = lib()
    M, N, K = 2048, 5120, 1024
    p = q4.gemm_plan(M, N, K)
    assert p["tile_rows"] > 256 and p["persistent"] and p["splits"] == 1, p
    x, wq = case(9900, M, N, K, outlier_blocks=0.05)
    xd, wd = x_dev(x), wq_dev(wq)
    y = q4.gemm(xd, wd, N, K)
    check_full(y, x, wq, N, K)
    assert torch.equal(q4.gemm(xd, wd, N, K), y)
    assert torch.equal(q4.matmul(xd, wd, N, K), y)
    assert q4.device_error() == 0


def test_gemm_one_wave_short_tiles_every_output():
    """M = 512 against 40 weight tiles takes three x tiles of 176 rows (the
    last ragged, 160 rows) in one wave: every output against the oracle,
    with fp32 and bf16 y."""
    q4 = lib()
    M, N, K = 512, 5120, 1024
    assert q4.gemm_plan(M, N, K)["tile_rows"] < 256
    x, wq = case(9910, M, N, K, act_outliers=0.01)
    xd, wd = x_dev(x), wq_dev(wq)
    y = q4.matmul(xd, wd, N, K)
    check_full(y, x, wq, N, K)
    assert torch.equal(q4.matmul(xd, wd, N, K, out_dtype=torch.bfloat16), y.to(torch.bfloat16))
    assert q4.device_error() == 0


def test_persistent_gemm_every_output():
    """The persistent GEMM (one CTA per SM taking tiles in turn, the
    accumulator drained by separate epilogue warps while the next tile's
    copies and dequantisation run): ragged M and N, two or three tiles per
    CTA; every output against the oracle, bitwise repeatable, and equal to
    the dispatcher's result."""
    q4 = lib()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    M, N, K = 500, 128 * (sms + 1) + 72, 512
    assert q4.gemm_plan(M, N, K)["persistent"]
    x, wq = case(9700, M, N, K, outlier_blocks=0.05, act_outliers=0.01)
    xd, wd = x_dev(x), wq_dev(wq)
    y = q4.gemm(xd, wd, N, K)
    check_full(y, x, wq, N, K)
    assert torch.equal(q4.gemm(xd, wd, N, K), y)
    assert torch.equal(q4.matmul(xd, wd, N, K), y)
    y16 = q4.matmul(xd, wd, N, K, out_dtype=torch.bfloat16)
    assert torch.equal(y16, y.to(torch.bfloat16))
    assert q4.device_error() == 0


def test_persistent_gemm_split_k():
    """The persistent GEMM over (tile, K split) units: the down shape at
    M = 1000 (four 256-row x tiles, K split four ways): sampled outputs
    against the oracle, bitwise repeatable."""
    q4 = lib()
    M, N, K = 1000, 5120, 17408
    p = q4.gemm_plan(M, N, K)
    assert p["persistent"] and p["splits"] > 1, p
    x, wq = case(9800, M, N, K, outlier_blocks=0.05, act_outliers=0.01)
    xd, wd = x_dev(x), wq_dev(wq)
    y = q4.gemm(xd, wd, N, K)
    check_sampled(y, x, wq, N, K, seed=3)
    assert torch.equal(q4.gemm(xd, wd, N, K), y)
    assert q4.device_error() == 0
