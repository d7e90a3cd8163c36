"""Shared helpers for the GPU tests: device transfer of the seeded inputs and
the comparison with the oracle."""
import numpy as np
import torch

import oracle


def lib():
    from q4_weight_only_gb300 import build
    build.build()
    import q4_weight_only_gb300 as q4
    return q4


def x_dev(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def wq_dev(wq: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(wq)).cuda()


def check_full(y_gpu: torch.Tensor, x_bits, wq, N, K):
    y_ref, absum = oracle.get().matmul(x_bits, wq, N, K)
    r = oracle.check(y_gpu.double().cpu().numpy(), y_ref, absum)
    assert r["ok"], r
    return r


def check_sampled(y_gpu: torch.Tensor, x_bits, wq, N, K, count=2048, seed=0, rel_l2=True):
    """Compare at `count` seeded (m, n) positions (plus the four corners)."""
    M = x_bits.shape[0]
    rng = np.random.default_rng(seed)
    ms = np.concatenate([rng.integers(0, M, count), [0, 0, M - 1, M - 1]])
    ns = np.concatenate([rng.integers(0, N, count), [0, N - 1, 0, N - 1]])
    y_ref, absum = oracle.get().matmul_sampled(x_bits, wq, N, K, ms, ns)
    sel = y_gpu[torch.from_numpy(ms).cuda(), torch.from_numpy(ns).cuda()].double().cpu().numpy()
    r = oracle.check(sel, y_ref, absum)
    assert r["ok"], r
    return r
