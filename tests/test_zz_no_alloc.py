"""fp8q_gemm_ws_static: the GEMM with its stream-K scratch in a fixed array
inside the library, for callers that cannot allocate device memory (e.g. a
plugin interface handed only its input and output buffers, or a path that
must not take cudaMalloc's implicit synchronization).

Both entry points run the same deterministic split of the K loop across SMs
(partials added in SM order), so on two calls in a row the static-scratch
result must equal fp8q_gemm_ws's bit for bit -- which also shows the shared
array is left usable by the first call -- and both must be within the GEMM
tolerance of the oracle's exact result.

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


def _bits(C):
    return C.view(torch.int16) if C.dtype == torch.bfloat16 else C.view(torch.int32)


@pytest.mark.parametrize("M,N,K,gran,out", [
    (256, 512, 8192, 128, torch.float32),    # 4 tiles of 64 K-blocks: every tile split across SMs
    (384, 768, 8192, 1, torch.float32),      # per-column B scales (the Wgrad form), 9 tiles x 64 K-blocks
    (256, 512, 8192, 128, torch.bfloat16),   # BF16 output through the same split
])
def test_static_scratch_matches_workspace_entry_point(M, N, K, gran, out):
    import fine_grained_fp8_quantize_b300 as f
    # the split only runs (and only then touches the scratch) when there are
    # at least as many K-blocks as SMs and the tiles leave the wave idle
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    tiles = ((M + 127) // 128) * ((N + 255) // 256)
    assert tiles * (K // 128) >= sms and tiles < sms
    rng = np.random.default_rng(M * 3 + N + K + gran)
    Aq, Bq = _codes(rng, (M, K)), _codes(rng, (N, K))
    sA = _scales(rng, (K // 128, M))
    sB = _scales(rng, (N // 128, K // 128)) if gran == 128 else _scales(rng, (K // 128, N))
    dA, dsA, dB, dsB = (torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in (Aq, sA, Bq, sB))

    ws = f.gemm_workspace()
    ref = torch.empty(M, N, dtype=out, device="cuda")
    f.fp8q_gemm_ws(dA, dsA, dB, dsB, ref, gran, ws)
    torch.cuda.synchronize()
    status_ok()
    exact, absref, _ = oracle.gemm(Aq, sA, Bq, sB, sb_gran=gran)
    check_gemm(gemm_out_to_f64(ref), exact, absref, out == torch.bfloat16, "workspace entry point")

    for call in range(2):
        C = torch.full((M, N), float("nan"), dtype=out, device="cuda")
        f.fp8q_gemm_ws_static(dA, dsA, dB, dsB, C, gran)
        torch.cuda.synchronize()
        status_ok()
        assert torch.equal(_bits(C), _bits(ref)), "static scratch, call %d: differs from fp8q_gemm_ws" % call
        check_gemm(gemm_out_to_f64(C), exact, absref, out == torch.bfloat16, "static scratch, call %d" % call)
