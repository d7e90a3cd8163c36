"""Shapes at the edges of what one launch holds, against the oracle.

* Tall matrices with one or two rows of x: the CUDA-core decode keeps each
  CTA's per-row partial sums in shared memory, so past a few hundred
  thousand rows (at K = 16384) the call runs as several launches over row
  ranges, each writing its columns of y with the full row stride.
* K past 65536 with one or two rows of x: x no longer fits shared memory,
  and the call takes the tensor-core decode (x streamed in binary16 tiles).
The tall cases use random Q4_0 blocks generated on the device (uniform
codes, binary16 scales of a typical magnitude) and compare a seeded sample
of rows in full; the long-K cases compare every output.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_common import check_full, lib, wq_dev, x_dev
from q4_weight_only_gb300 import synth

pytestmark = pytest.mark.gpu


def random_q4_0(N, K, seed):
    """Q4_0 bytes [N, K/32*18] on the device: codes uniform, scales ~ N(0, 2e-3) in binary16."""
    g = torch.Generator(device="cuda").manual_seed(seed)
    nb = K // 32
    wq = torch.randint(0, 256, (N, nb, 18), dtype=torch.uint8, device="cuda", generator=g)
    d = (torch.randn((N, nb), device="cuda", generator=g) * 2e-3).half()
    wq[:, :, 0:2] = d.view(torch.uint8).view(N, nb, 2)
    return wq.view(N, nb * 18)


def check_rows(y, x_bits, wq, K, rows):
    """y[:, rows] against the oracle on those weight rows."""
    rows = np.unique(rows)
    sub = wq[torch.from_numpy(rows).cuda()].cpu().numpy()
    y_ref, absum = oracle.get().matmul(x_bits, sub, len(rows), K)
    got = y[:, torch.from_numpy(rows).cuda()].double().cpu().numpy()
    r = oracle.check(got, y_ref, absum)
    assert r["ok"], r


@pytest.mark.parametrize("N,K", [(400_000, 16384),    # integer-dot kernel (K % 1024 == 0)
                                 (300_000, 16640)])   # binary16 kernel
@pytest.mark.parametrize("M", [1, 2])
def test_tall_matrix_runs_as_several_launches(M, N, K):
    q4 = lib()
    wq = random_q4_0(N, K, seed=N + K)
    rng = np.random.default_rng(N + M)
    x_bits = synth.to_bf16_bits(rng.standard_normal((M, K), dtype=np.float32))
    y = q4.matmul(x_dev(x_bits), wq, N, K)
    # rows spread over the whole matrix (every launch's range) plus both ends
    rows = np.concatenate([rng.integers(0, N, 192), np.linspace(0, N - 1, 64).astype(np.int64), [0, N - 1]])
    check_rows(y, x_bits, wq, K, rows)
    assert q4.device_error() == 0
    del wq
    torch.cuda.empty_cache()


@pytest.mark.parametrize("K", [65536, 65792, 131072])
@pytest.mark.parametrize("M", [1, 2])
def test_long_k_one_or_two_rows(M, K):
    """K = 65536 is the longest the CUDA-core decode holds; past it the call
    takes the tensor-core decode, with scratch from q4_0_matmul_workspace_bytes."""
    q4 = lib()
    N = 300
    w, x = synth.small_case(9900 + M + K // 256, M, N, K, outlier_block_frac=0.05, act_outlier_frac=0.01)
    wq = oracle.get().quantize(w)
    need = int(q4.lib().q4_0_matmul_workspace_bytes(M, N, K))
    assert (need > 0) == (K > 65536)
    xd, wd = x_dev(x), wq_dev(wq)
    check_full(q4.matmul(xd, wd, N, K), x, wq, N, K)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
    assert torch.equal(q4.matmul(xd, wd, N, K, workspace=ws), q4.matmul(xd, wd, N, K))
    assert q4.device_error() == 0
