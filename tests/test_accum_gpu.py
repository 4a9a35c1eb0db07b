"""The accumulation-precision diagnostic (fp8q_gemm_unpromoted): the whole K
accumulated inside the tensor core, against the oracle and against the
promoted GEMM.  The pages attribute a maximum relative error near 2% at an
inner dimension of 4096 to limited tensor-core accumulation ("Eliminate
Deepseek Ai News For Good", the accumulation-precision sentence); these tests
pin what the diagnostic computes, not that figure."""
import numpy as np
import pytest
import torch

import oracle
from helpers import check_gemm, gemm_out_to_f64, status_ok

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def f():
    import fine_grained_fp8_quantize_b300 as f
    return f


def _codes(rng, shape):
    c = rng.integers(0, 256, shape).astype(np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x3F
    return c


def test_single_kblock_equals_promoted_bitwise(f):
    # K = 128: one K-block, so "promote once with unit scales" and
    # "accumulate in the tensor core" are the same FP32 value
    rng = np.random.default_rng(11)
    M, N, K = 200, 384, 128
    A = torch.from_numpy(_codes(rng, (M, K))).cuda()
    B = torch.from_numpy(_codes(rng, (N, K))).cuda()
    one_a = torch.ones(K // 128, M, device="cuda")
    one_b = torch.ones(N // 128, K // 128, device="cuda")
    Cu = torch.empty(M, N, dtype=torch.float32, device="cuda")
    f.fp8q_gemm_unpromoted(A, B, Cu)
    Cp = f.gemm(A, one_a, B, one_b, out_dtype=torch.float32)
    torch.cuda.synchronize()
    status_ok()
    assert torch.equal(Cu.view(torch.int32), Cp.view(torch.int32))


@pytest.mark.parametrize("M,N,K", [(128, 256, 1024), (257, 512, 4096)])
def test_unpromoted_close_to_exact(f, M, N, K):
    rng = np.random.default_rng(M + N + K)
    Aq, Bq = _codes(rng, (M, K)), _codes(rng, (N, K))
    Cu = torch.empty(M, N, dtype=torch.float32, device="cuda")
    f.fp8q_gemm_unpromoted(torch.from_numpy(Aq).cuda(), torch.from_numpy(Bq).cuda(), Cu)
    torch.cuda.synchronize()
    status_ok()
    ones_a = np.ones((K // 128, M), np.float32)
    ones_b = np.ones((N // 128, K // 128), np.float32)
    ex, ab, _ = oracle.gemm(Aq, ones_a, Bq, ones_b)
    # whatever the tensor core's internal accumulation, it is a sum of the
    # same products: within the GEMM tolerance of the exact result
    check_gemm(gemm_out_to_f64(Cu), ex, ab, False, "unpromoted %dx%dx%d" % (M, N, K))
