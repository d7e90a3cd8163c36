"""Pins for the Q4_0 oracle: checks against values and facts fixed outside it.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError when the
oracle disagrees with a hand-derived value, IEEE 754 (through numpy/torch's
own converters), exact rational arithmetic, or an invariant of the block
definition.  ``test_oracle_pins.py`` runs them on the real oracle;
``test_oracle_mutants.py`` runs the fast ones on builds with one planted
mistake each and requires at least one to fail.
"""
import json
import os
from fractions import Fraction

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "q4_0_blocks.json")


def golden():
    with open(GOLDEN) as f:
        return json.load(f)


def golden_block_weights(block):
    w = np.zeros((1, 32), dtype=np.float32)
    for idx, lit in block["w"].items():
        w[0, int(idx)] = np.float32(float(lit))
    return w


def _bf16_bits_of(value: float) -> int:
    """bf16 bits of a value that is exactly representable in bf16."""
    f = np.array([value], dtype=np.float32)
    bits = int(f.view(np.uint32)[0])
    assert bits & 0xFFFF == 0, "not exactly representable in bf16"
    return bits >> 16


def _fraction_f16(bits: int) -> Fraction:
    return Fraction(float(np.array([bits], dtype=np.uint16).view(np.float16)[0]))


def _fraction_bf16(bits: int) -> Fraction:
    return Fraction(float(np.array([bits << 16], dtype=np.uint32).view(np.float32)[0]))


# ------------------------------------------------------------------ golden

def pin_golden_blocks(o):
    for b in golden()["blocks"]:
        got = o.quantize(golden_block_weights(b)).tobytes().hex()
        assert got == b["bytes"], f"{b['name']}: {got} != {b['bytes']}"


# Codes of the 'rounding_half_away_clamp_and_nibble_order' block, by hand
# (see its derivation in the golden file): elements 0..31.
ROUNDING_BLOCK_CODES = [0, 11, 5, 9, 7, 10, 6, 15, 15, 0, 8, 8, 8, 8, 8, 8,
                        11, 5, 8, 8, 8, 8, 8, 8, 8, 8, 8, 8, 8, 8, 8, 8]


def pin_golden_unpack(o):
    b = {x["name"]: x for x in golden()["blocks"]}["rounding_half_away_clamp_and_nibble_order"]
    wq = np.frombuffer(bytes.fromhex(b["bytes"]), dtype=np.uint8).reshape(1, 18)
    codes, dbits = o.unpack(wq, 1, 32)
    assert codes[0].tolist() == ROUNDING_BLOCK_CODES, codes[0].tolist()
    assert int(dbits[0, 0]) == 0x3C00


def pin_golden_dequant(o):
    """The grid block decodes back to its weights exactly."""
    b = {x["name"]: x for x in golden()["blocks"]}["grid_round_trip"]
    wq = np.frombuffer(bytes.fromhex(b["bytes"]), dtype=np.uint8).reshape(1, 18)
    w = o.dequantize(wq, 1, 32)
    assert np.array_equal(w, golden_block_weights(b).astype(np.float64)), w


def pin_golden_matmul(o):
    g = golden()
    blocks = {x["name"]: x for x in g["blocks"]}
    for mm in g["matmuls"]:
        wq = np.frombuffer(bytes.fromhex(blocks[mm["block"]]["bytes"]), dtype=np.uint8).reshape(1, 18)
        x = np.zeros((1, 32), dtype=np.uint16)
        if "fill" in mm["x"]:
            x[:] = _bf16_bits_of(float(mm["x"]["fill"]))
        for k, v in mm["x"].get("entries", {}).items():
            x[0, int(k)] = _bf16_bits_of(float(v))
        y, _ = o.matmul(x, wq, 1, 32)
        assert y[0, 0] == float(mm["y"]), f"{mm['name']}: {y[0, 0]} != {mm['y']}"


# ------------------------------------------------------------ IEEE formats

def pin_f16_decode_exhaustive(o):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = o.f16_bits_to_f64(bits)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def pin_bf16_decode_exhaustive(o):
    import torch
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    got = o.bf16_bits_to_f64(bits)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def _check_f16_encode(o, f32):
    import torch
    got = o.f32_to_f16_array(f32)
    ref = torch.from_numpy(f32).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(f32)
    bad = (got != ref) & ~nan
    assert not bad.any(), f"{int(bad.sum())} mismatches, first input bits 0x{int(f32.view(np.uint32)[np.argmax(bad)]):08x}"
    # NaN stays NaN
    if nan.any():
        g = got[nan]
        assert np.all(((g & 0x7C00) == 0x7C00) & ((g & 0x3FF) != 0))


def pin_f16_encode_sampled(o, n=1 << 22, seed=7):
    """Every binary32 exponent with random and boundary mantissas."""
    rng = np.random.default_rng(seed)
    u = rng.integers(0, 1 << 32, size=n, dtype=np.uint64).astype(np.uint32)
    # the mantissa bits that decide binary16 rounding: exact ties and +-1 around them
    exps = np.arange(256, dtype=np.uint32) << 23
    tails = np.array([0x0000, 0x0FFF, 0x1000, 0x1001, 0x1FFF, 0x2000, 0x3000, 0x7FFFFF], dtype=np.uint32)
    grid = (exps[:, None] | tails[None, :]).ravel()
    u = np.concatenate([u, grid, grid | 0x80000000])
    _check_f16_encode(o, u.view(np.float32))
    # numpy's converter as a second, independent reference on a subset
    sub = u[: 1 << 16].view(np.float32)
    with np.errstate(over="ignore"):
        ref = sub.astype(np.float16).view(np.uint16)
    got = o.f32_to_f16_array(sub)
    assert np.array_equal(got[~np.isnan(sub)], ref[~np.isnan(sub)])


def pin_f16_encode_exhaustive(o, chunk_log2=24):
    """All 2^31 non-negative binary32 patterns (the sign is a separate bit),
    in chunks written into one reused buffer."""
    step = 1 << chunk_log2
    ramp = np.arange(step, dtype=np.uint32)
    u = np.empty(step, dtype=np.uint32)
    for start in range(0, 1 << 31, step):
        np.add(ramp, np.uint32(start), out=u)
        _check_f16_encode(o, u.view(np.float32))


# --------------------------------------------------------------- invariants

def _random_blocks(seed, nblocks=4096):
    rng = np.random.default_rng(seed)
    parts = [
        rng.normal(0, 0.02, (nblocks, 32)),
        rng.normal(0, 0.2, (nblocks, 32)),
        rng.uniform(-3, 3, (nblocks, 32)),
        rng.standard_cauchy((nblocks, 32)) * 0.01,
        rng.normal(0, 1, (nblocks, 32)) * (10.0 ** rng.integers(-4, 3, (nblocks, 1))),
    ]
    w = np.concatenate(parts).astype(np.float32)
    return w.reshape(1, -1)  # one long row of blocks


def pin_roundtrip_invariant(o, seed=11):
    """|w - d*(q-8)| <= |d| (1/2 + 2^-8) / (1 - 2^-11) for unclamped codes (q < 15),
    <= |d| (1 + 2^-8) / (1 - 2^-11) for q = 15 (clamped side); the max-|w|
    element takes code 0; sign(d) = -sign(max element); |d| is max|w|/8 to
    binary16 precision."""
    w = _random_blocks(seed)
    K = w.shape[1]
    wq = o.quantize(w)
    codes, dbits = o.unpack(wq, 1, K)
    d = o.f16_bits_to_f64(dbits.ravel())
    wb = w.reshape(-1, 32).astype(np.float64)
    qb = codes.reshape(-1, 32).astype(np.float64)
    err = np.abs(wb - d[:, None] * (qb - 8))
    ad = np.abs(d)[:, None]
    tight = ad * (0.5 + 2.0 ** -8) / (1 - 2.0 ** -11)
    loose = ad * (1.0 + 2.0 ** -8) / (1 - 2.0 ** -11)
    normal = (np.abs(d) >= 2.0 ** -14)[:, None]
    assert np.all(err[(qb < 15) & normal] <= np.broadcast_to(tight, err.shape)[(qb < 15) & normal])
    assert np.all(err[(qb == 15) & normal] <= np.broadcast_to(loose, err.shape)[(qb == 15) & normal])
    imax = np.argmax(np.abs(wb), axis=1)  # numpy argmax: first index of the max
    rows = np.arange(wb.shape[0])
    assert np.all(qb[rows, imax] == 0)
    wmax = wb[rows, imax]
    assert np.all(np.sign(d) == -np.sign(wmax))
    nz = normal[:, 0]
    rel = np.abs(np.abs(d[nz]) - np.abs(wmax[nz]) / 8) / (np.abs(wmax[nz]) / 8)
    assert np.all(rel <= 2.0 ** -11)


def pin_grid_roundtrip(o, seed=13):
    """Weights already on a power-of-two grid d*(c-8) with c[0] = 0 come back exactly."""
    rng = np.random.default_rng(seed)
    nblk = 2048
    c = rng.integers(0, 16, (nblk, 32))
    c[:, 0] = 0
    scale = 2.0 ** rng.integers(-12, 4, (nblk, 1))
    w = (scale * (c - 8)).astype(np.float32).reshape(1, -1)
    wq = o.quantize(w)
    back = o.dequantize(wq, 1, w.shape[1])
    assert np.array_equal(back, w.astype(np.float64))


# ------------------------------------------------------------------ matmul

def _random_q4_bytes(rng, N, K):
    """Random valid blocks: finite normal binary16 d of either sign, random codes."""
    nb = K // 32
    exp = rng.integers(1, 25, (N, nb))           # keep |d| well inside the normal range
    man = rng.integers(0, 1024, (N, nb))
    sign = rng.integers(0, 2, (N, nb))
    dbits = (sign << 15) | (exp << 10) | man
    wq = np.empty((N, nb, 18), dtype=np.uint8)
    wq[..., 0] = dbits & 0xFF
    wq[..., 1] = dbits >> 8
    wq[..., 2:] = rng.integers(0, 256, (N, nb, 16))
    return wq.reshape(N, nb * 18)


def _exact_weights(wq, N, K):
    """The block definition, read straight from the bytes, as Fractions."""
    nb = K // 32
    b = wq.reshape(N, nb, 18)
    W = [[None] * K for _ in range(N)]
    for n in range(N):
        for j in range(nb):
            d = _fraction_f16(int(b[n, j, 0]) | (int(b[n, j, 1]) << 8))
            for i in range(16):
                byte = int(b[n, j, 2 + i])
                W[n][32 * j + i] = d * ((byte & 15) - 8)
                W[n][32 * j + i + 16] = d * ((byte >> 4) - 8)
    return W


def pin_fraction_bruteforce(o, seed=17, M=2, N=3, K=64):
    """Exact rational sums vs the fp64 oracle (error <= K * 2^-53 * sum |w x|)."""
    rng = np.random.default_rng(seed)
    wq = _random_q4_bytes(rng, N, K)
    xf = rng.normal(0, 1, (M, K)).astype(np.float32)
    x = (xf.view(np.uint32) >> 16).astype(np.uint16)        # truncation: any bf16 is fine
    y, a = o.matmul(x, wq, N, K)
    W = _exact_weights(wq, N, K)
    for m in range(M):
        xs = [_fraction_bf16(int(v)) for v in x[m]]
        for n in range(N):
            exact = sum(W[n][k] * xs[k] for k in range(K))
            absum = sum(abs(W[n][k] * xs[k]) for k in range(K))
            tol = float(absum) * K * 2.0 ** -52
            assert abs(y[m, n] - float(exact)) <= tol, (m, n, y[m, n], float(exact))
            assert abs(a[m, n] - float(absum)) <= tol, (m, n, a[m, n], float(absum))


def pin_one_hot(o, seed=19, N=5, K=96):
    """x = e_k for every k: y[k, n] is exactly the decoded weight w[n, k]."""
    rng = np.random.default_rng(seed)
    wq = _random_q4_bytes(rng, N, K)
    x = np.zeros((K, K), dtype=np.uint16)
    np.fill_diagonal(x, 0x3F80)  # bf16 1.0
    y, _ = o.matmul(x, wq, N, K)
    W = _exact_weights(wq, N, K)
    expect = np.array([[float(W[n][k]) for n in range(N)] for k in range(K)])
    assert np.array_equal(y, expect)


def pin_linearity(o, seed=23, M=3, N=4, K=128):
    """y(x1 + x2) = y(x1) + y(x2) for x1, x2 whose sum is exact in bf16."""
    rng = np.random.default_rng(seed)
    wq = _random_q4_bytes(rng, N, K)
    a = rng.integers(-8, 8, (M, K)).astype(np.float32) / 16
    b = rng.integers(-8, 8, (M, K)).astype(np.float32) / 16
    to_bits = lambda v: (v.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    y1, _ = o.matmul(to_bits(a), wq, N, K)
    y2, _ = o.matmul(to_bits(b), wq, N, K)
    y12, abs12 = o.matmul(to_bits(a + b), wq, N, K)
    assert np.all(np.abs(y12 - (y1 + y2)) <= 4 * K * 2.0 ** -52 * (abs12 + 1e-300) + 1e-300)


def pin_sampled_matches_full(o, seed=29, M=4, N=37, K=256):
    rng = np.random.default_rng(seed)
    wq = _random_q4_bytes(rng, N, K)
    x = (rng.normal(0, 1, (M, K)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    y, a = o.matmul(x, wq, N, K)
    ms = rng.integers(0, M, 50)
    ns = rng.integers(0, N, 50)
    ys, as_ = o.matmul_sampled(x, wq, N, K, ms, ns)
    assert np.array_equal(ys, y[ms, ns]) and np.array_equal(as_, a[ms, ns])


FAST_PINS = [pin_golden_blocks, pin_golden_unpack, pin_golden_dequant, pin_golden_matmul,
             pin_f16_encode_sampled, pin_roundtrip_invariant, pin_grid_roundtrip,
             pin_fraction_bruteforce, pin_one_hot, pin_linearity, pin_sampled_matches_full]
