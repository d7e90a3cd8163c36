"""q4_0_gemm_noalloc against q4_0_gemm (GPU).

q4_0_gemm_noalloc serves callers that cannot allocate device memory: its
scratch is a fixed array inside the library.  Called straight through the C
ABI, twice in a row on different inputs, it must give what the workspace
entry point gives, within the tolerance the other tests use, and it must
refuse sizes its array cannot hold; sampled rows are also checked against the
oracle.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_common import lib, wq_dev, x_dev
from q4_weight_only_gb300 import synth

pytestmark = pytest.mark.gpu


def _call_noalloc(q4, xd, wd, y, M, N, K):
    st = torch.cuda.current_stream().cuda_stream
    return q4.lib().q4_0_gemm_noalloc(xd.data_ptr(), wd.data_ptr(), y.data_ptr(), M, N, K, st)


def test_noalloc_matches_gemm_on_two_calls():
    q4 = lib()
    o = oracle.get()
    cases = [(300, 520, 1536, 11), (2048, 384, 5120, 12)]  # second one: 20 MiB of scratch
    for M, N, K, seed in cases:
        w, x = synth.small_case(seed, M, N, K, outlier_block_frac=0.05)
        wq = o.quantize(w)
        xd, wd = x_dev(x), wq_dev(wq)
        ref = q4.gemm(xd, wd, N, K)                   # existing entry point, caller workspace
        y = torch.full((M, N), float("nan"), device="cuda")
        assert _call_noalloc(q4, xd, wd, y, M, N, K) == q4.OK
        torch.cuda.synchronize()
        rows = np.arange(0, M, max(1, M // 64))
        y_ref, absum = o.matmul(x[rows], wq, N, K)
        got = y[torch.from_numpy(rows).cuda()].double().cpu().numpy()
        exp = ref[torch.from_numpy(rows).cuda()].double().cpu().numpy()
        # against the oracle, and against the workspace entry point (which
        # may split K and so sum in another order: tolerance, not bits)
        r = oracle.check(got, y_ref, absum)
        assert r["ok"], r
        r = oracle.check(got, exp, absum)
        assert r["ok"], r
    assert q4.device_error() == 0


def test_noalloc_refuses_oversize():
    q4 = lib()
    K = 1024
    M = (32 * 1024 * 1024) // (2 * K) + 1               # one row more than the array holds
    xd = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    wd = torch.zeros((128, K // 32 * 18), dtype=torch.uint8, device="cuda")
    y = torch.zeros((M, 128), device="cuda")
    assert _call_noalloc(q4, xd, wd, y, M, 128, K) == q4.ERR_WORKSPACE
