"""fp8q_gemm_ws_static: the GEMM with its stream-K scratch in a fixed array
inside the library, for callers that cannot allocate device memory (e.g. a
plugin interface handed only its input and output buffers, or a path that
must not take cudaMalloc's implicit synchronization).  Its output must match
fp8q_gemm_ws (caller workspace) on two calls in a row, so the second call
also shows that the shared array is left in a usable state.

This file sorts last so a run that stops at the first failure has already
run every other test."""
import numpy as np
import pytest
import torch

import oracle
from helpers import check_gemm, gemm_out_to_f64, status_ok

pytestmark = pytest.mark.gpu


def _codes(rng, shape):
    c = rng.integers(0, 256, shape).astype(np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x3F  # no NaN codes
    return c


def _scales(rng, shape):
    return (2.0 ** rng.uniform(-10, 3, shape)).astype(np.float32)


@pytest.mark.parametrize("M,N,K,gran", [
    (256, 512, 8192, 128),   # 4 tiles of 64 K-blocks: every tile split across SMs
    (384, 768, 2048, 1),     # per-column B scales (the Wgrad form)
])
def test_static_scratch_matches_workspace_entry_point(M, N, K, gran):
    import fine_grained_fp8_quantize_b300 as f
    rng = np.random.default_rng(M * 3 + N + K + gran)
    Aq, Bq = _codes(rng, (M, K)), _codes(rng, (N, K))
    sA = _scales(rng, (K // 128, M))
    sB = _scales(rng, (N // 128, K // 128)) if gran == 128 else _scales(rng, (K // 128, N))
    dA, dsA, dB, dsB = (torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in (Aq, sA, Bq, sB))

    ws = f.gemm_workspace()
    ref = torch.empty(M, N, dtype=torch.float32, device="cuda")
    f.fp8q_gemm_ws(dA, dsA, dB, dsB, ref, gran, ws)
    torch.cuda.synchronize()
    status_ok()
    _, absref, _ = oracle.gemm(Aq, sA, Bq, sB, sb_gran=gran)
    ref64 = gemm_out_to_f64(ref)

    for call in range(2):
        C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        f.fp8q_gemm_ws_static(dA, dsA, dB, dsB, C, gran)
        torch.cuda.synchronize()
        status_ok()
        # within the GEMM tolerance of the workspace entry point's result
        check_gemm(gemm_out_to_f64(C), ref64, absref, False, "static scratch, call %d" % call)
