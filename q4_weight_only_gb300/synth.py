"""Seeded synthetic inputs for the Q4_0 matmul workloads.

This module only draws random numbers: it holds none of the Q4_0 arithmetic
(no quantizer, no unpack, no matmul), so both the CUDA path and the CPU
oracle can take their inputs from it.

Workloads (27B-class dense-layer shapes, K the reduction dimension):

* ``pr1``      W [256, 1024] ~ N(0, 0.02) fp32; x [1, 1024] ~ N(0, 1) -> bf16;
               one generator seeded 0, W drawn before x.
* ``decode``   M = 1 over (N, K) in SHAPES; W ~ N(0, 0.02); x ~ N(0, 1);
               seed 100 + shape index (W then x).
* ``batched``  M in (4, 8, 16, 32) over the same shapes and the same W as
               ``decode``; x ~ N(0, 1) with 1 % of entries scaled by 20
               (activation outliers); seed 200 + 10 * shape + M index.
* ``prefill``  M in (512, 2048, 8192); W ~ N(0, 0.02) except 5 % of the
               32-weight blocks redrawn from N(0, 0.2); x ~ N(0, 1);
               W seed 300 + shape index, x seed 400 + 10 * shape + M index.
* ``sweep``    64 layers of the four shapes, drawn on the device (see
               ``device_layer_weights``).

All draws use numpy's PCG64 (bit-identical on x86-64 and aarch64); bf16
activations are the round-to-nearest-even bf16 of the fp32 draws.
"""
import numpy as np

SHAPES = {
    "qkv": (7168, 5120),
    "o": (5120, 5120),
    "gate_up": (34816, 5120),
    "down": (5120, 17408),
}
SHAPE_ORDER = ("qkv", "o", "gate_up", "down")
BATCHED_M = (4, 8, 16, 32)
PREFILL_M = (512, 2048, 8192)
N_LAYERS = 64
WEIGHT_STD = 0.02
OUTLIER_BLOCK_STD = 0.2
OUTLIER_BLOCK_FRAC = 0.05
ACT_OUTLIER_FRAC = 0.01
ACT_OUTLIER_SCALE = 20.0


def generator(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def weights(gen: np.random.Generator, N: int, K: int, std: float = WEIGHT_STD,
            outlier_block_frac: float = 0.0, outlier_std: float = OUTLIER_BLOCK_STD) -> np.ndarray:
    """fp32 [N, K] ~ N(0, std); optionally a Bernoulli fraction of the
    32-wide blocks along K redrawn from N(0, outlier_std)."""
    w = gen.standard_normal((N, K), dtype=np.float32)
    w *= np.float32(std)
    if outlier_block_frac > 0.0:
        mask = gen.random((N, K // 32)) < outlier_block_frac
        rows, blks = np.nonzero(mask)
        alt = gen.standard_normal((rows.size, 32), dtype=np.float32) * np.float32(outlier_std)
        view = w.reshape(N, K // 32, 32)
        view[rows, blks, :] = alt
    return w


def activations_f32(gen: np.random.Generator, M: int, K: int, outlier_frac: float = 0.0,
                    outlier_scale: float = ACT_OUTLIER_SCALE) -> np.ndarray:
    """fp32 [M, K] ~ N(0, 1); optionally a Bernoulli fraction of entries x scale."""
    x = gen.standard_normal((M, K), dtype=np.float32)
    if outlier_frac > 0.0:
        mask = gen.random((M, K)) < outlier_frac
        x[mask] *= np.float32(outlier_scale)
    return x


def to_bf16_bits(x_f32: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even bf16 of fp32 values, returned as uint16 bits."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x_f32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def pr1():
    """(W fp32 [256, 1024], x bf16 bits [1, 1024])."""
    g = generator(0)
    w = weights(g, 256, 1024)
    x = to_bf16_bits(activations_f32(g, 1, 1024))
    return w, x


def decode_weights(shape: str) -> np.ndarray:
    N, K = SHAPES[shape]
    return weights(generator(100 + SHAPE_ORDER.index(shape)), N, K)


def decode(shape: str):
    """(W fp32 [N, K], x bf16 bits [1, K]) for M = 1 decode on one shape."""
    N, K = SHAPES[shape]
    g = generator(100 + SHAPE_ORDER.index(shape))
    w = weights(g, N, K)
    x = to_bf16_bits(activations_f32(g, 1, K))
    return w, x


def batched_x(shape: str, M: int) -> np.ndarray:
    """bf16 bits [M, K] with activation outliers, for batched decode."""
    _, K = SHAPES[shape]
    g = generator(200 + 10 * SHAPE_ORDER.index(shape) + BATCHED_M.index(M))
    return to_bf16_bits(activations_f32(g, M, K, outlier_frac=ACT_OUTLIER_FRAC))


def prefill_weights(shape: str) -> np.ndarray:
    N, K = SHAPES[shape]
    return weights(generator(300 + SHAPE_ORDER.index(shape)), N, K,
                   outlier_block_frac=OUTLIER_BLOCK_FRAC)


def prefill_x(shape: str, M: int) -> np.ndarray:
    _, K = SHAPES[shape]
    g = generator(400 + 10 * SHAPE_ORDER.index(shape) + PREFILL_M.index(M))
    return to_bf16_bits(activations_f32(g, M, K))


def small_case(seed: int, M: int, N: int, K: int, outlier_block_frac: float = 0.0,
               act_outlier_frac: float = 0.0):
    """(W fp32 [N, K], x bf16 bits [M, K]) for the small parity cases."""
    g = generator(seed)
    w = weights(g, N, K, outlier_block_frac=outlier_block_frac)
    x = to_bf16_bits(activations_f32(g, M, K, outlier_frac=act_outlier_frac))
    return w, x


def device_layer_weights(layer: int, shape: str, device="cuda"):
    """fp32 [N, K] ~ N(0, 0.02) drawn on the device with a per-(layer, shape)
    seeded torch generator (the 64-layer sweep is too large to draw on the host)."""
    import torch
    N, K = SHAPES[shape]
    g = torch.Generator(device=device)
    g.manual_seed(10_000 + 10 * layer + SHAPE_ORDER.index(shape))
    w = torch.empty((N, K), dtype=torch.float32, device=device)
    w.normal_(0.0, WEIGHT_STD, generator=g)
    return w
