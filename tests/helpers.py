"""Shared helpers of the GPU parity tests (test code only)."""
import numpy as np
import torch

import oracle
import synth

# GEMM acceptance: |C - C*| <= 2e-3 * sum_k |a_dq * b_dq| per element for FP32
# output, plus one BF16 rounding (half an ulp: 2^-8 relative) for BF16 output.
GEMM_RTOL_ABS = 2e-3
BF16_ROUND = 2.0 ** -8


def host_bits(t):
    """Device/host BF16 tensor -> numpy uint16 bits; FP32 -> numpy float32."""
    if t.dtype == torch.bfloat16:
        return synth.bf16_bits(t)
    return t.detach().cpu().numpy()


def to_np(t):
    return t.detach().cpu().numpy()


def status_ok():
    import fine_grained_fp8_quantize_b300 as f
    st = f.fp8q_get_device_status()
    assert st == 0, "device status %d (%s)" % (st, f.fp8q_status_string(st))


def check_gemm(C, exact, absref, out_bf16, what=""):
    """C: GPU result (float64 numpy), exact/absref: oracle (same shape)."""
    err = np.abs(C - exact)
    tol = GEMM_RTOL_ABS * absref
    if out_bf16:
        tol = tol * (1 + BF16_ROUND) + BF16_ROUND * np.abs(exact)
    bad = err > tol
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError("%s: %d of %d outside tolerance; first at %s: gpu %r exact %r absref %r"
                             % (what, bad.sum(), bad.size, tuple(i), C[tuple(i)], exact[tuple(i)],
                                absref[tuple(i)]))
    # the result is a genuine approximation, not a loose bound met by zeros
    nz = absref > 0
    if nz.any():
        assert np.median(err[nz] / absref[nz]) < 1e-3, what
    return float((err[nz] / absref[nz]).max()) if nz.any() else 0.0


def gemm_out_to_f64(C):
    return C.detach().float().cpu().numpy().astype(np.float64)


def sample_points(M, N, tile_m=128, tile_n=256, seed=0):
    """One full row per M-tile and one full column per N-tile (plus the last
    row and column) -> (m_idx, n_idx) of every element on those lines."""
    rng = np.random.default_rng(seed)
    rows = sorted({int(min(M - 1, t * tile_m + rng.integers(0, tile_m))) for t in range((M + tile_m - 1) // tile_m)}
                  | {M - 1})
    cols = sorted({int(min(N - 1, t * tile_n + rng.integers(0, tile_n))) for t in range((N + tile_n - 1) // tile_n)}
                  | {N - 1})
    mi = np.concatenate([np.full(N, r, np.int64) for r in rows] + [np.arange(M, dtype=np.int64) for _ in cols])
    ni = np.concatenate([np.arange(N, dtype=np.int64) for _ in rows] + [np.full(M, c, np.int64) for c in cols])
    return mi, ni
