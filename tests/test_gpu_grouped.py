"""q4_0_matmul_grouped: several independent problems in one call.  Problems
the grouped decode takes (M = 1, K % 1024 == 0) run in persistent launches
of up to eight; every result must equal its one-problem q4_0_matmul_ex call
bit for bit, and the oracle on a sample."""
import numpy as np
import pytest
import torch

import oracle
from gpu_common import check_sampled, lib
from q4_weight_only_gb300 import synth

pytestmark = pytest.mark.gpu


def x_bits_of(x: torch.Tensor) -> np.ndarray:
    return x.view(torch.int16).cpu().numpy().view(np.uint16)


def random_x(M, K, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return torch.randn((M, K), device="cuda", generator=g).to(torch.bfloat16)


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("M", [1, 2])
def test_layer_matrices_in_one_launch(M, out_dtype):
    """The four layer matrices (QKV, O, gate+up, down) as one group."""
    q4 = lib()
    shapes = synth.SHAPE_ORDER
    Ns = [synth.SHAPES[s][0] for s in shapes]
    Ks = [synth.SHAPES[s][1] for s in shapes]
    wqs = [q4.quantize(synth.device_layer_weights(0, s)) for s in shapes]
    xs = [random_x(M, K, 40 + i) for i, K in enumerate(Ks)]
    ys = q4.matmul_grouped(xs, wqs, Ns, Ks, out_dtype=out_dtype)
    for x, wq, y, N, K in zip(xs, wqs, ys, Ns, Ks):
        assert torch.equal(y, q4.matmul(x, wq, N, K, out_dtype=out_dtype))
    if out_dtype == torch.float32:
        for i in (1, 3):   # O and down against the oracle
            check_sampled(ys[i], x_bits_of(xs[i]), wqs[i].cpu().numpy(), Ns[i], Ks[i], count=512, seed=i)
    assert q4.device_error() == 0


def test_mixed_group_matches_single_calls():
    """Problems the grouped decode cannot take (K % 1024 != 0, K % 256 != 0,
    K past 65536) run one by one inside the same call, in order."""
    q4 = lib()
    M = 1
    probs = [(5120, 5120), (300, 1280), (1000, 2048), (200, 96), (257, 131072), (129, 1024), (4099, 3072)]
    xs, wqs, Ns, Ks = [], [], [], []
    for i, (N, K) in enumerate(probs):
        w, x = synth.small_case(700 + i, M, N, K)
        xs.append(torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda())
        wqs.append(torch.from_numpy(oracle.get().quantize(w)).cuda())
        Ns.append(N)
        Ks.append(K)
    ys = q4.matmul_grouped(xs, wqs, Ns, Ks)
    for x, wq, y, N, K in zip(xs, wqs, ys, Ns, Ks):
        assert torch.equal(y, q4.matmul(x, wq, N, K)), (N, K)
    assert q4.device_error() == 0


def test_more_problems_than_one_launch_holds():
    """Ten eligible problems: the library splits them into launches of at
    most eight; the results still equal the one-problem calls."""
    q4 = lib()
    M = 1
    xs, wqs, Ns, Ks = [], [], [], []
    for i in range(10):
        N, K = 257 + 64 * i, 1024 * (1 + i % 3)
        g = torch.Generator(device="cuda").manual_seed(900 + i)
        w = torch.randn((N, K), device="cuda", generator=g) * 0.02
        wqs.append(q4.quantize(w))
        xs.append(random_x(M, K, 950 + i))
        Ns.append(N)
        Ks.append(K)
    ys = q4.matmul_grouped(xs, wqs, Ns, Ks)
    for x, wq, y, N, K in zip(xs, wqs, ys, Ns, Ks):
        assert torch.equal(y, q4.matmul(x, wq, N, K)), (N, K)
    check_sampled(ys[9], x_bits_of(xs[9]), wqs[9].cpu().numpy(), Ns[9], Ks[9], count=256)
    assert q4.device_error() == 0


def test_batched_rows_fall_back_to_single_calls():
    """M = 16 is not a grouped-decode size: every problem is its own call
    (M = 2 in test_layer_matrices_in_one_launch likewise)."""
    q4 = lib()
    M = 16
    Ns, Ks = [700, 300], [2048, 5120]
    xs = [random_x(M, K, 60 + i) for i, K in enumerate(Ks)]
    g = torch.Generator(device="cuda").manual_seed(61)
    wqs = [q4.quantize(torch.randn((N, K), device="cuda", generator=g) * 0.02) for N, K in zip(Ns, Ks)]
    ys = q4.matmul_grouped(xs, wqs, Ns, Ks)
    for x, wq, y, N, K in zip(xs, wqs, ys, Ns, Ks):
        assert torch.equal(y, q4.matmul(x, wq, N, K))
