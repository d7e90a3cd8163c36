"""The device unpack and scale apply, bit for bit (GPU, through the C ABI).

With x one-hot (row m of x is v times the unit vector e_k), y[m][n] is one
decoded weight times v, so a swapped nibble, a wrong byte of the scale, a
permuted k position or a mis-scaled block shows up as a wrong value rather
than as a small error inside the tolerance.  The Q4_0 format ("Vertical
disaggregation: maximizing model throughput on heterogeneous silicon",
section "Every cycle counts: custom kernels": one shared format, nibble
unpack and scale apply) fixes every decoded weight w = d (q - 8):

  * the integer-dot decode (M <= 2) multiplies exact integer sums by
    d * 2^(e-14) in fp32, so y = w v exactly (w v has at most 17 significant
    bits);
  * the binary16 decode for general K (M <= 2, K % 1024 != 0) scales x and
    the codes by powers of two, so y = w v exactly too;
  * the tensor-core paths (batched decode, GEMM) dequantise to binary16 with
    one rounding, so y = RN16(w) v exactly.

The expected values come from the oracle alone: its dequantize (w, exact in
fp64) and its binary16 encoder (RN16), both pinned against IEEE 754.  The
matrices mix every scale class the kernels treat differently: |d| >= 2^-10
(the d / 16 route), normal |d| < 2^-10 and subnormal d (the shift route),
d = 0, and |d| >= 64; both signs; every code value.  Rows in alternate
128-row weight tiles hold large scales only, so that both the stages taken
through the d / 16 route and the mixed stages taken through the shift route
are checked.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_common import lib, wq_dev

pytestmark = pytest.mark.gpu


def q4_matrix(seed, N, K):
    """Q4_0 bytes [N, K/32*18] with uniform random codes and binary16 scales
    drawn from five classes (see the module docstring)."""
    rng = np.random.default_rng(seed)
    nb = K // 32
    cls = rng.integers(0, 5, size=(N, nb))
    # the tensor-core kernels pick the d / 16 route for a whole stage of a
    # warp's 32 rows when every scale in it is large: rows in even 128-row
    # tiles draw large scales only, so that route is taken there, and the
    # odd tiles mix all five classes
    large_only = (np.arange(N) // 128 % 2 == 0)[:, None]
    cls = np.where(large_only, np.where(rng.random((N, nb)) < 0.5, 0, 4), cls)
    exp = np.select([cls == 0, cls == 1, cls == 4], [rng.integers(5, 15, size=(N, nb)),
                                                      rng.integers(1, 5, size=(N, nb)),
                                                      rng.integers(21, 27, size=(N, nb))], 0)
    mant = rng.integers(0, 1024, size=(N, nb))
    mant = np.where(cls == 2, rng.integers(1, 1024, size=(N, nb)), mant)   # subnormal: mantissa != 0
    mant = np.where(cls == 3, 0, mant)                                        # zero scale
    sign = rng.integers(0, 2, size=(N, nb)) << 15
    dbits = (sign | (exp << 10) | mant).astype(np.uint16)
    blocks = np.empty((N, nb, 18), dtype=np.uint8)
    blocks[..., 0] = dbits & 0xFF
    blocks[..., 1] = dbits >> 8
    blocks[..., 2:] = rng.integers(0, 256, size=(N, nb, 16), dtype=np.uint8)
    return blocks.reshape(N, nb * 18)


def expected(wq, N, K, rounded16):
    """E[n][k] = w (exact) or RN16(w), from the oracle."""
    o = oracle.get()
    w = o.dequantize(wq, N, K)                    # exact d (q - 8) in fp64
    if not rounded16:
        return w
    w32 = w.astype(np.float32)
    assert np.array_equal(w32.astype(np.float64), w)  # w is exact in fp32
    bits = o.f32_to_f16_array(w32)
    table = o.f16_bits_to_f64(np.arange(65536, dtype=np.uint16))
    return table[bits]


def one_hot_x(K, v):
    """bf16 [K, K]: row k is v e_k."""
    return (torch.eye(K, dtype=torch.float32) * v).to(torch.bfloat16).cuda()


def starts(K, M, stride=None):
    """First x rows of calls of exactly M rows that cover 0..K-1 (the last
    call is moved back so that every call keeps M rows, and with it its
    path); `stride` > M skips rows."""
    return sorted({min(k, K - M) for k in range(0, K, stride or M)})


def run_rows(fn, X, rows, N, K, step):
    """y rows [k, k + step) from calls on x rows [k, k + step) of X."""
    Y = torch.full((K, N), float("nan"), dtype=torch.float32, device="cuda")
    for k in rows:
        Y[k:k + step] = fn(X[k:k + step])
    torch.cuda.synchronize()
    return Y.double().cpu().numpy()


def assert_exact(Y, E, v, rows, step, K, what):
    got = np.concatenate([Y[k:k + step] for k in rows])
    want = np.concatenate([(E[:, k:k + step] * v).T for k in rows])
    bad = got != want
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} outputs differ, first at {np.argwhere(bad)[0]}"


@pytest.mark.parametrize("v", [1.0, -0.75])
def test_one_hot_integer_dot_decode(v):
    """M = 1 and M = 2 through the integer-dot decode: every (n, k) exact."""
    q4 = lib()
    N, K = 256, 1024
    wq = q4_matrix(11, N, K)
    wd = wq_dev(wq)
    E = expected(wq, N, K, rounded16=False)
    X = one_hot_x(K, v)
    for M in (1, 2):
        rows = starts(K, M)
        Y = run_rows(lambda xs: q4.gemv(xs, wd, N, K), X, rows, N, K, M)
        assert_exact(Y, E, v, rows, M, K, f"integer-dot decode M={M}")
    assert q4.device_error() == 0


def test_one_hot_general_k_decode():
    """M <= 2 with K % 1024 != 0 takes the binary16 decode kernel: exact."""
    q4 = lib()
    N, K = 200, 1280
    wq = q4_matrix(12, N, K)
    wd = wq_dev(wq)
    E = expected(wq, N, K, rounded16=False)
    X = one_hot_x(K, 1.0)
    for M in (1, 2):
        rows = starts(K, M, stride=3 if M == 1 else None)
        Y = run_rows(lambda xs: q4.gemv(xs, wd, N, K), X, rows, N, K, M)
        assert_exact(Y, E, 1.0, rows, M, K, f"binary16 decode M={M}")
    assert q4.device_error() == 0


@pytest.mark.parametrize("v", [1.0, -0.75])
def test_one_hot_tensor_core_decode(v):
    """3 <= M <= 64 through the tcgen05 batched decode: every (n, k) equals
    RN16(w) v, for tiles of 16, 32 and 64 rows, and for M = 3."""
    q4 = lib()
    N, K = 300, 1024
    wq = q4_matrix(13, N, K)
    wd = wq_dev(wq)
    E = expected(wq, N, K, rounded16=True)
    X = one_hot_x(K, v)
    for M in (3, 16, 32, 64):
        rows = starts(K, M)
        Y = run_rows(lambda xs: q4.gemv(xs, wd, N, K), X, rows, N, K, M)
        assert_exact(Y, E, v, rows, M, K, f"tensor-core decode M={M}")
    assert q4.device_error() == 0


@pytest.mark.parametrize("v", [1.0, -0.75])
def test_one_hot_gemm(v):
    """The tcgen05 GEMM: x = v I (M = K = 1024, four 256-row tiles) checks
    every (n, k) in one call; M = 272 (one tall tile, a second MMA per k
    step) and M = 64 (the split-K partial-tile sum) cover the other tile
    forms."""
    q4 = lib()
    N, K = 384, 1024
    wq = q4_matrix(14, N, K)
    wd = wq_dev(wq)
    E = expected(wq, N, K, rounded16=True)
    X = one_hot_x(K, v)
    for M in (K, 272, 64):
        rows = starts(K, M)
        Y = run_rows(lambda xs: q4.gemm(xs, wd, N, K), X, rows, N, K, M)
        assert_exact(Y, E, v, rows, M, K, f"GEMM M={M}")
    assert q4.device_error() == 0



def test_one_hot_persistent_gemm():
    """x = I (M = K = 512, two 256-row x tiles) against a matrix of enough
    weight tiles that the persistent GEMM runs: every (n, k) equals
    RN16(w) exactly."""
    q4 = lib()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    N, K = 128 * (sms + 1) + 72, 512
    assert q4.gemm_plan(K, N, K)["persistent"]
    wq = q4_matrix(15, N, K)
    wd = wq_dev(wq)
    E = expected(wq, N, K, rounded16=True)
    X = one_hot_x(K, 1.0)
    Y = run_rows(lambda xs: q4.gemm(xs, wd, N, K), X, [0], N, K, K)
    assert_exact(Y, E, 1.0, [0], K, K, "persistent GEMM")
    assert q4.device_error() == 0


def test_one_hot_persistent_tall_gemm():
    """x = v I through tall x tiles (M = 272, a second MMA per k step) with
    more weight tiles than SMs, so that the persistent form runs: every
    (n, k) equals RN16(w) v exactly."""
    q4 = lib()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    N, K, M = 128 * (sms + 8) + 40, 1024, 272
    p = q4.gemm_plan(M, N, K)
    assert p["persistent"] and p["tile_rows"] == 272, p
    wq = q4_matrix(16, N, K)
    wd = wq_dev(wq)
    E = expected(wq, N, K, rounded16=True)
    X = one_hot_x(K, -0.75)
    rows = starts(K, M)
    Y = run_rows(lambda xs: q4.gemm(xs, wd, N, K), X, rows, N, K, M)
    assert_exact(Y, E, -0.75, rows, M, K, "persistent tall GEMM")
    assert q4.device_error() == 0

def test_scale_classes_present():
    """The test matrices hold every scale class the kernels distinguish."""
    o = oracle.get()
    N, K = 256, 1024
    _, dbits = o.unpack(q4_matrix(11, N, K), N, K)
    e = (dbits >> 10) & 0x1F
    assert ((e >= 5) & (e < 15)).any() and ((e >= 1) & (e < 5)).any()
    assert ((e == 0) & ((dbits & 0x3FF) != 0)).any() and ((dbits & 0x7FFF) == 0).any()
    assert (e >= 21).any() and (dbits >> 15).any() and not (dbits >> 15).all()
