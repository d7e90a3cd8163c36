"""Device quantizer: codes and scales bit-exact with the oracle."""
import numpy as np
import pytest
import torch

import oracle
import pins
from gpu_common import lib
from q4_weight_only_gb300 import synth

pytestmark = pytest.mark.gpu


def gpu_quantize(w: np.ndarray) -> np.ndarray:
    q4 = lib()
    return q4.quantize(torch.from_numpy(np.ascontiguousarray(w)).cuda()).cpu().numpy()


def test_golden_blocks_on_device():
    for b in pins.golden()["blocks"]:
        got = gpu_quantize(pins.golden_block_weights(b)).tobytes().hex()
        assert got == b["bytes"], b["name"]


def test_pr1_bit_exact():
    w, _ = synth.pr1()
    assert np.array_equal(gpu_quantize(w), oracle.get().quantize(w))


@pytest.mark.parametrize("shape", synth.SHAPE_ORDER)
def test_decode_weights_bit_exact(shape):
    w = synth.decode_weights(shape)
    assert np.array_equal(gpu_quantize(w), oracle.get().quantize(w))


@pytest.mark.parametrize("shape", ["o", "down"])
def test_prefill_weights_bit_exact(shape):
    w = synth.prefill_weights(shape)
    assert np.array_equal(gpu_quantize(w), oracle.get().quantize(w))


def test_edge_blocks_bit_exact():
    """Ties, zeros, -0, clamps, subnormal and large scales, ragged N."""
    rng = np.random.default_rng(5)
    blocks = [
        np.zeros(32), -np.zeros(32), np.full(32, 1.0), np.full(32, -1.0),
        np.r_[1.0, -1.0, np.zeros(30)], np.r_[-1.0, 1.0, np.zeros(30)],
        np.r_[np.zeros(31), 3.0], np.arange(32) - 16.0, (np.arange(32) - 16.0) * 1e-7,
        rng.normal(0, 1e-6, 32), rng.normal(0, 1e4, 32), rng.normal(0, 1e-30, 32),
        np.r_[-8.0, 7.5, -7.5, 2.5, -2.5, 0.5, -0.5, np.zeros(25)],
    ]
    for _ in range(200):
        c = rng.integers(0, 16, 32).astype(np.float64)
        c[rng.integers(0, 32)] = 0
        blocks.append((c - 8) * rng.choice([0.25, 0.1, 3.0, 1e-3]) + rng.choice([0, 1e-9]))
    w = np.stack(blocks).astype(np.float32).reshape(-1, 32)
    for N in (1, 3, w.shape[0]):
        sub = w[:N]
        assert np.array_equal(gpu_quantize(sub), oracle.get().quantize(sub))
    wide = w[: (w.shape[0] // 8) * 8].reshape(-1, 256)
    assert np.array_equal(gpu_quantize(wide), oracle.get().quantize(wide))


@pytest.mark.parametrize("layer", [0, 63])
def test_sweep_layers_bit_exact(layer):
    """The 64-layer sweep draws its weights on the device and quantizes them
    there; its first and last layers, all four shapes, match the oracle's
    quantizer on the same values bit for bit."""
    q4 = lib()
    for shape in synth.SHAPE_ORDER:
        w = synth.device_layer_weights(layer, shape)
        got = q4.quantize(w).cpu().numpy()
        assert np.array_equal(got, oracle.get().quantize(w.cpu().numpy())), shape
        del w
