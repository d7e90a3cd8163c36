"""Q4_0 oracle: a plain, slow CPU reference (TEST INFRASTRUCTURE ONLY).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It wraps the plain-C library built from
``oracle/q4_0_oracle.c`` (fp64 dequantize-then-matmul, fp32 quantizer
decision) with numpy in/out.  It shares nothing with the CUDA library.

Sources followed (see the C file for the full statement):
"Vertical disaggregation: maximizing model throughput on heterogeneous
silicon", section "Every cycle counts: custom kernels" (one shared Q4_0
format, deterministic output, nibble unpack / dot product / scale apply), and
the Q4_0 block definition this library fixes (32 weights, fp16 d, 16 code
bytes, w = d*(q-8), low nibble = element j, high nibble = element j+16).

Pins: every function here is checked by ``tests/test_oracle_pins.py`` against
values fixed by hand, by IEEE 754, by exact rational arithmetic or by
invariants; ``tests/test_oracle_mutants.py`` shows each planted mistake fails
at least one pin.
"""
import ctypes
import os

import numpy as np

from . import build as _build

QK = 32
BLOCK_BYTES = 18

_libs = {}


def _load(mutant: int = 0, out_dir: str = None):
    key = (mutant, out_dir)
    if key not in _libs:
        path = _build.build(mutant=mutant, out_dir=out_dir)
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        lib.oracle_f32_to_f16_bits.argtypes = [ctypes.c_float]
        lib.oracle_f32_to_f16_bits.restype = ctypes.c_uint16
        lib.oracle_f16_bits_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_f16_bits_to_f64.restype = ctypes.c_double
        lib.oracle_bf16_bits_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_bits_to_f64.restype = ctypes.c_double
        lib.oracle_f32_to_f16_array.argtypes = [P, P, I64]
        lib.oracle_quantize.argtypes = [P, P, I64, I64]
        lib.oracle_unpack.argtypes = [P, P, P, I64, I64]
        lib.oracle_dequantize.argtypes = [P, P, I64, I64]
        lib.oracle_matmul.argtypes = [P, P, P, P, I64, I64, I64]
        lib.oracle_matmul_sampled.argtypes = [P, P, I64, I64, I64, P, P, I64, P, P]
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_mutant.restype = ctypes.c_int
        _libs[key] = lib
    return _libs[key]


class Oracle:
    """numpy-facing wrapper around one build (the real one or a mutant)."""

    def __init__(self, mutant: int = 0, out_dir: str = None):
        self.lib = _load(mutant, out_dir)

    # -- binary16 / bfloat16 ----------------------------------------------
    def f32_to_f16_bits(self, values):
        v = np.ascontiguousarray(values, dtype=np.float32).ravel()
        return np.array([self.lib.oracle_f32_to_f16_bits(float(f)) for f in v], dtype=np.uint16)

    def f32_to_f16_array(self, values):
        v = np.ascontiguousarray(values, dtype=np.float32)
        out = np.empty(v.shape, dtype=np.uint16)
        self.lib.oracle_f32_to_f16_array(v.ctypes.data, out.ctypes.data, v.size)
        return out

    def f16_bits_to_f64(self, bits):
        b = np.ascontiguousarray(bits, dtype=np.uint16).ravel()
        return np.array([self.lib.oracle_f16_bits_to_f64(int(h)) for h in b], dtype=np.float64)

    def bf16_bits_to_f64(self, bits):
        b = np.ascontiguousarray(bits, dtype=np.uint16).ravel()
        return np.array([self.lib.oracle_bf16_bits_to_f64(int(h)) for h in b], dtype=np.float64)

    # -- quantizer / decoder ------------------------------------------------
    def quantize(self, w):
        """fp32 [N, K] -> uint8 [N, K/32*18] Q4_0 blocks."""
        w = np.ascontiguousarray(w, dtype=np.float32)
        N, K = w.shape
        if K % QK:
            raise ValueError("K must be a multiple of 32")
        out = np.empty((N, K // QK * BLOCK_BYTES), dtype=np.uint8)
        self.lib.oracle_quantize(w.ctypes.data, out.ctypes.data, N, K)
        return out

    def unpack(self, wq, N, K):
        """Q4_0 bytes -> (codes uint8 [N, K] in 0..15, d bits uint16 [N, K/32])."""
        wq = np.ascontiguousarray(wq, dtype=np.uint8)
        codes = np.empty((N, K), dtype=np.uint8)
        dbits = np.empty((N, K // QK), dtype=np.uint16)
        self.lib.oracle_unpack(wq.ctypes.data, codes.ctypes.data, dbits.ctypes.data, N, K)
        return codes, dbits

    def dequantize(self, wq, N, K):
        """Q4_0 bytes -> fp64 [N, K], w = d*(q-8) exactly."""
        wq = np.ascontiguousarray(wq, dtype=np.uint8)
        w = np.empty((N, K), dtype=np.float64)
        self.lib.oracle_dequantize(wq.ctypes.data, w.ctypes.data, N, K)
        return w

    # -- matmul -------------------------------------------------------------
    def matmul(self, x_bits, wq, N, K):
        """x: bf16 bits uint16 [M, K]; returns (y fp64 [M, N], abssum fp64 [M, N])."""
        x = np.ascontiguousarray(x_bits, dtype=np.uint16)
        wq = np.ascontiguousarray(wq, dtype=np.uint8)
        M = x.shape[0]
        y = np.empty((M, N), dtype=np.float64)
        a = np.empty((M, N), dtype=np.float64)
        self.lib.oracle_matmul(x.ctypes.data, wq.ctypes.data, y.ctypes.data, a.ctypes.data, M, N, K)
        return y, a

    def matmul_sampled(self, x_bits, wq, N, K, ms, ns):
        """The matmul evaluated only at the (ms[i], ns[i]) pairs."""
        x = np.ascontiguousarray(x_bits, dtype=np.uint16)
        wq = np.ascontiguousarray(wq, dtype=np.uint8)
        ms = np.ascontiguousarray(ms, dtype=np.int64)
        ns = np.ascontiguousarray(ns, dtype=np.int64)
        y = np.empty(len(ms), dtype=np.float64)
        a = np.empty(len(ms), dtype=np.float64)
        self.lib.oracle_matmul_sampled(x.ctypes.data, wq.ctypes.data, x.shape[0], N, K,
                                       ms.ctypes.data, ns.ctypes.data, len(ms),
                                       y.ctypes.data, a.ctypes.data)
        return y, a

    def threads(self):
        return int(self.lib.oracle_num_threads())


_default = None


def get() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default


# Tolerances for a floating-point result against the oracle: per element,
# |y - y_ref| <= ABS_FRAC * sum_k |w[n,k] x[m,k]|; globally, the relative L2
# error ||y - y_ref|| / ||y_ref|| <= REL_L2.
ABS_FRAC = 1e-2
REL_L2 = 2e-3


def check(y, y_ref, abssum, abs_frac: float = ABS_FRAC, rel_l2: float = REL_L2):
    """Compare a result with the oracle under the two tolerance rules."""
    y = np.asarray(y, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    abssum = np.asarray(abssum, dtype=np.float64)
    err = np.abs(y - y_ref)
    bound = abs_frac * abssum
    finite = bool(np.all(np.isfinite(y)))
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(bound > 0, err / np.where(bound > 0, bound, 1), np.where(err > 0, np.inf, 0.0))
    max_ratio = float(ratio.max()) if ratio.size else 0.0
    nref = float(np.linalg.norm(y_ref))
    rel = float(np.linalg.norm(y - y_ref) / nref) if nref > 0 else float(np.linalg.norm(y - y_ref))
    ok = finite and max_ratio <= 1.0 and rel <= rel_l2
    return {"ok": ok, "max_ratio": max_ratio, "rel_l2": rel, "finite": finite}
