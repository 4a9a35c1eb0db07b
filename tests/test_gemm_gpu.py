"""GPU parity of the block-scaled FP8 GEMM (dense, Wgrad per-column scales,
MoE grouped) against the CPU oracle, through the C ABI.

Acceptance per element: |C - C*| <= 2e-3 * sum_k |a_dq * b_dq| against the
oracle's exact result C* (FP32 output), plus one BF16 rounding for BF16
output.  FP8 GEMMs with FP32 promotion every 128 K: "Eliminate Deepseek Ai
News For Good", the MMA-precision passage; inprokorea.com page, the
accumulation-interval passage."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import check_gemm, gemm_out_to_f64, host_bits, sample_points, status_ok, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def f():
    import fine_grained_fp8_quantize_b300 as f
    return f


def rand_codes(rng, shape):
    c = rng.integers(0, 256, shape).astype(np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x3F
    return c


def rand_scales(rng, shape):
    return (2.0 ** rng.uniform(-10, 3, shape)).astype(np.float32)


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run_dense(f, Aq, sA, Bq, sB, out, gran=128):
    C = f.gemm(dev(Aq), dev(sA), dev(Bq), dev(sB), out_dtype=out, sb_gran_n=gran)
    torch.cuda.synchronize()
    status_ok()
    return gemm_out_to_f64(C)


@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
def test_tiny_end_to_end_128x128x512(f, out):
    # A BF16 128x512 N(0,1) with 1% entries x100, B BF16 512x128 N(0, 0.02^2):
    # quantize on the GPU (A 1x128, B 128x128), GEMM on the GPU, compare
    # every output with the oracle run on the same BF16 inputs.
    A, Bt = synth.tiny_gemm_inputs(device="cuda", seed=0)
    qa, sa, _, _ = f.quantize_act(A)
    qb, sb = f.quantize_weight(Bt)
    C = f.gemm(qa, sa, qb, sb, out_dtype=out)
    torch.cuda.synchronize()
    status_ok()
    oqa, osa = oracle.quantize_act_rows(host_bits(A))
    oqb, osb = oracle.quantize_weight(host_bits(Bt))
    assert np.array_equal(to_np(qa), oqa) and np.array_equal(to_np(qb), oqb)
    ex, ab, pg = oracle.gemm(oqa, osa, oqb, osb)
    check_gemm(gemm_out_to_f64(C), ex, ab, out == torch.bfloat16, "tiny")


@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (300, 640, 1024), (1, 128, 256), (257, 384, 384)])
@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
def test_dense_random_codes(f, M, N, K, out):
    rng = np.random.default_rng(M * 7 + N + K)
    Aq, Bq = rand_codes(rng, (M, K)), rand_codes(rng, (N, K))
    sA = rand_scales(rng, (K // 128, M))
    sB = rand_scales(rng, (N // 128, K // 128))
    C = run_dense(f, Aq, sA, Bq, sB, out)
    ex, ab, _ = oracle.gemm(Aq, sA, Bq, sB)
    check_gemm(C, ex, ab, out == torch.bfloat16, "dense %dx%dx%d" % (M, N, K))


def test_dense_many_waves(f):
    # 16 x 16 = 256 tiles > one wave of persistent CTAs
    rng = np.random.default_rng(5)
    M, N, K = 2048, 4096, 256
    Aq, Bq = rand_codes(rng, (M, K)), rand_codes(rng, (N, K))
    sA = rand_scales(rng, (K // 128, M))
    sB = rand_scales(rng, (N // 128, K // 128))
    C = run_dense(f, Aq, sA, Bq, sB, torch.float32)
    mi, ni = sample_points(M, N, seed=1)
    ex, ab, _ = oracle.gemm_points(Aq, sA, Bq, sB, mi, ni)
    check_gemm(C[mi, ni], ex, ab, False, "many waves")


def test_dense_zero_rows_is_noop(f):
    Aq = torch.empty(0, 256, dtype=torch.uint8, device="cuda")
    sA = torch.empty(2, 0, dtype=torch.float32, device="cuda")
    Bq = torch.zeros(128, 256, dtype=torch.uint8, device="cuda")
    sB = torch.ones(1, 2, dtype=torch.float32, device="cuda")
    C = f.gemm(Aq, sA, Bq, sB)
    torch.cuda.synchronize()
    assert C.shape == (0, 128)


@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (256, 384, 1024), (200, 640, 512)])
def test_wgrad_per_column_scales(f, M, N, K, out):
    # every output element; half N-tiles and a ragged M-tile; both output
    # types (the per-column variant stores from its own register layout)
    rng = np.random.default_rng(N + K)
    Aq, Bq = rand_codes(rng, (M, K)), rand_codes(rng, (N, K))
    sA = rand_scales(rng, (K // 128, M))
    sB = rand_scales(rng, (K // 128, N))
    C = run_dense(f, Aq, sA, Bq, sB, out, gran=1)
    ex, ab, _ = oracle.gemm(Aq, sA, Bq, sB, sb_gran=1)
    check_gemm(C, ex, ab, out == torch.bfloat16, "wgrad")


def test_fprop_full_size_4096x18432x7168(f):
    # X BF16 4096x7168 N(0,1), 0.1% entries x1e3; W BF16 18432x7168 N(0,0.02^2)
    X, W = synth.fprop_inputs(device="cuda")
    qx, sx, _, _ = f.quantize_act(X)
    qw, sw = f.quantize_weight(W)
    C = f.gemm(qx, sx, qw, sw, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    status_ok()
    mi, ni = sample_points(4096, 18432, seed=3)
    hqx, hsx, hqw, hsw = to_np(qx), to_np(sx), to_np(qw), to_np(sw)
    # the operands themselves are bit-exact: every row of X (codes and scale
    # bits); W is compared in full in test_quantize_full_gpu.py
    oq, os_ = oracle.quantize_act_rows(host_bits(X))
    assert np.array_equal(hqx, oq) and np.array_equal(hsx.view(np.uint32), os_.view(np.uint32))
    ex, ab, _ = oracle.gemm_points(hqx, hsx, hqw, hsw, mi, ni)
    check_gemm(gemm_out_to_f64(C)[mi, ni], ex, ab, True, "fprop full size")


def test_wgrad_full_size_2048x7168x8192(f):
    # dW = dY^T X: dY BF16 8192x2048 N(0,1e-6) with 0.5% x50, X BF16 8192x7168
    # N(0,1); both quantized 128x1 along the 8192 tokens; FP32 output
    dY, X = synth.wgrad_inputs(device="cuda")
    _, _, qdy, sdy = f.quantize_act(dY, row=False, col=True)
    _, _, qx, sx = f.quantize_act(X, row=False, col=True)
    C = f.gemm(qdy, sdy, qx, sx, out_dtype=torch.float32, sb_gran_n=1)
    torch.cuda.synchronize()
    status_ok()
    mi, ni = sample_points(2048, 7168, seed=4)
    ex, ab, _ = oracle.gemm_points(to_np(qdy), to_np(sdy), to_np(qx), to_np(sx), mi, ni, sb_gran=1)
    check_gemm(gemm_out_to_f64(C)[mi, ni], ex, ab, False, "wgrad full size")


def test_dgrad_with_transposed_weight(f):
    # dX = dY . W: dY 1x128-quantized rows, W's transposed codes/scales
    dY = synth.matrix(41, 1, 256, 384, 1e-3, entry_frac=5e-3, entry_scale=50.0, device="cuda")
    W = synth.matrix(42, 2, 384, 512, 0.02, device="cuda")        # [N_out=384, K_in=512]
    qdy, sdy, _, _ = f.quantize_act(dY)
    _, _, qwt, swt = f.quantize_weight(W, transposed=True)         # [512, 384], [4, 3]
    C = f.gemm(qdy, sdy, qwt, swt, out_dtype=torch.float32)
    torch.cuda.synchronize()
    status_ok()
    ex, ab, _ = oracle.gemm(to_np(qdy), to_np(sdy), to_np(qwt), to_np(swt))
    check_gemm(gemm_out_to_f64(C), ex, ab, False, "dgrad")
    ref = (dY.double() @ W.double()).cpu().numpy()
    assert np.abs(gemm_out_to_f64(C) - ref).max() < 0.15 * np.abs(ref).max()


def test_dgrad_full_size_4096x7168x18432(f):
    # dX = dY . W, the third Linear GEMM in FP8 (dssusan.co.kr page, the
    # Figure 6 passage): dY BF16 4096x18432 (N(0,1e-6), 0.5% x50) in 1x128
    # groups over the 18432 output features; W the Fprop weight BF16
    # 18432x7168, whose transposed 128x128-block codes [7168][18432] and
    # scales [56][144] are the B operand.  M 4096, N 7168, K 18432, BF16 out.
    dY = synth.matrix(5, 1, 4096, 18432, 1e-3, entry_frac=5e-3, entry_scale=50.0, device="cuda")
    _, W = synth.fprop_inputs(device="cuda", M=128)
    qdy, sdy, _, _ = f.quantize_act(dY)
    _, _, qwt, swt = f.quantize_weight(W, transposed=True)
    del W
    C = f.gemm(qdy, sdy, qwt, swt, out_dtype=torch.bfloat16)
    # 896 tiles = 6.05 waves: with a workspace the tail goes through stream-K
    # (the scale-ring variant with split tiles)
    Cs = f.gemm(qdy, sdy, qwt, swt, out_dtype=torch.bfloat16, workspace=f.gemm_workspace())
    torch.cuda.synchronize()
    status_ok()
    mi, ni = sample_points(4096, 7168, seed=6)
    ex, ab, _ = oracle.gemm_points(to_np(qdy), to_np(sdy), to_np(qwt), to_np(swt), mi, ni)
    check_gemm(gemm_out_to_f64(C)[mi, ni], ex, ab, True, "dgrad full size")
    check_gemm(gemm_out_to_f64(Cs)[mi, ni], ex, ab, True, "dgrad full size, stream-K")


def test_raster_groups_with_ragged_last_group(f):
    # A larger than 64 MiB of codes switches the dense GEMM to its grouped
    # tile order (16 M-tiles per group over all N-tiles).  M 2240 = 17.5
    # M-tiles: groups of 16 and 2, the last M-tile ragged; N 384: one full
    # and one half N-tile; K 30720 (240 K-blocks).  Random codes (no NaN) and
    # scales 2^U(-10,3); every output of one row per M-tile and one column
    # per N-tile is compared with the oracle.
    rng = np.random.default_rng(2240)
    M, N, K = 2240, 384, 30720
    assert M * K > 64 << 20
    Aq, Bq = rand_codes(rng, (M, K)), rand_codes(rng, (N, K))
    sA = rand_scales(rng, (K // 128, M))
    sB = rand_scales(rng, ((N + 127) // 128, K // 128))
    C = run_dense(f, Aq, sA, Bq, sB, torch.bfloat16)
    mi, ni = sample_points(M, N, seed=11)
    ex, ab, _ = oracle.gemm_points(Aq, sA, Bq, sB, mi, ni)
    check_gemm(C[mi, ni], ex, ab, True, "grouped raster order")


def test_tensor_core_partials_vs_pages_order():
    # Diagnostic of the tensor core's internal accumulation: the GPU result
    # (FP32 out, K = 7168 = 56 promotions) against the oracle's literal FP32
    # procedure of the pages (P_kb rounded to FP32, times fl32(sA*sB), added
    # in K-block order; "Eliminate Deepseek Ai News For Good", the
    # MMA-precision passage).  Both approximate the exact sum; if the tensor
    # core's 128-term partials were exact FP32 the two would differ only by
    # the promotion's FMA against separate roundings, about 56 ulps of the
    # running sum.  The bound 2e-5 * sum|ab| is 100x tighter than the parity
    # tolerance; the measured maximum is printed.
    import fine_grained_fp8_quantize_b300 as f
    rng = np.random.default_rng(7168)
    M, N, K = 256, 512, 7168
    Aq, Bq = rand_codes(rng, (M, K)), rand_codes(rng, (N, K))
    sA = rand_scales(rng, (K // 128, M))
    sB = rand_scales(rng, (N // 128, K // 128))
    C = run_dense(f, Aq, sA, Bq, sB, torch.float32)
    ex, ab, pg = oracle.gemm(Aq, sA, Bq, sB)
    d_pages = float((np.abs(C - pg.astype(np.float64)) / ab).max())
    d_exact = float((np.abs(C - ex) / ab).max())
    p_exact = float((np.abs(pg.astype(np.float64) - ex) / ab).max())
    print("max |C_gpu - C_pages|/sum|ab| = %.3g; |C_gpu - exact| %.3g; |C_pages - exact| %.3g"
          % (d_pages, d_exact, p_exact))
    assert d_pages <= 2e-5, d_pages


# ----------------------------------------------------------------- grouped

def run_grouped(f, Aq, sA, Bq, sB, off, out):
    C = f.grouped_gemm(dev(Aq), dev(sA), dev(Bq), dev(sB), dev(off.astype(np.int32)), out_dtype=out)
    torch.cuda.synchronize()
    status_ok()
    return gemm_out_to_f64(C)


@pytest.mark.parametrize("counts", [[0, 130, 1, 0, 77], [300], [0, 0, 5], [128, 128, 256, 1, 0, 129]])
@pytest.mark.parametrize("out", [torch.bfloat16, torch.float32])
def test_grouped_ragged_and_empty(f, counts, out):
    rng = np.random.default_rng(sum(counts) + len(counts))
    E, N, K = len(counts), 384, 256
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    T = int(off[-1])
    Aq = rand_codes(rng, (T, K))
    sA = rand_scales(rng, (K // 128, T))
    Bq = rand_codes(rng, (E, N, K))
    sB = rand_scales(rng, (E, N // 128, K // 128))
    C = run_grouped(f, Aq, sA, Bq, sB, off, out)
    for e in range(E):
        r0, r1 = off[e], off[e + 1]
        if r1 == r0:
            continue
        ex, ab, _ = oracle.gemm(Aq[r0:r1], np.ascontiguousarray(sA[:, r0:r1]), Bq[e], sB[e])
        check_gemm(C[r0:r1], ex, ab, out == torch.bfloat16, "expert %d" % e)


def test_grouped_many_tiles(f):
    rng = np.random.default_rng(99)
    counts = [0, 700, 3, 129, 0, 1000, 260, 0]
    E, N, K = len(counts), 1280, 384
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    T = int(off[-1])
    Aq = rand_codes(rng, (T, K))
    sA = rand_scales(rng, (K // 128, T))
    Bq = rand_codes(rng, (E, N, K))
    sB = rand_scales(rng, (E, N // 128, K // 128))
    C = run_grouped(f, Aq, sA, Bq, sB, off, torch.bfloat16)
    for e in range(E):
        r0, r1 = off[e], off[e + 1]
        if r1 == r0:
            continue
        mi, ni = sample_points(r1 - r0, N, seed=e)
        ex, ab, _ = oracle.gemm_points(Aq[r0:r1], np.ascontiguousarray(sA[:, r0:r1]), Bq[e], sB[e], mi, ni)
        check_gemm(C[r0:r1][mi, ni], ex, ab, True, "expert %d" % e)


def test_moe_full_size_256_experts(f):
    # 8192 tokens x 7168, 256 experts, top-8 of sigmoid(logit) + bias (skewed),
    # each expert 7168 -> 2048, BF16 out.  Quantize-before-dispatch with the
    # fused gather, one grouped GEMM; oracle on sampled rows/cols of the
    # busiest, the lightest and a middle expert.
    off, src = synth.moe_routing()
    counts = off[1:] - off[:-1]
    active = np.flatnonzero(counts)
    E, N, K = 256, 2048, 7168
    X, W = synth.moe_inputs(device="cuda", experts=[int(e) for e in active])
    qx, sx = f.quantize_act_gather(X, torch.from_numpy(src.astype(np.int32)).cuda())
    qw, sw = f.quantize_weight(W.view(E * N, K))
    qw = qw.view(E, N, K)
    sw = sw.view(E, N // 128, K // 128)
    C = f.grouped_gemm(qx, sx, qw, sw, torch.from_numpy(off.astype(np.int32)).cuda(), out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    status_ok()
    Ch = gemm_out_to_f64(C)
    hqx, hsx = to_np(qx), to_np(sx)
    order = active[np.argsort(counts[active])]
    for e in {int(order[-1]), int(order[0]), int(order[len(order) // 2])}:
        r0, r1 = int(off[e]), int(off[e + 1])
        mi, ni = sample_points(r1 - r0, N, seed=e)
        ex, ab, _ = oracle.gemm_points(hqx[r0:r1], np.ascontiguousarray(hsx[:, r0:r1]), to_np(qw[e]),
                                       to_np(sw[e]), mi, ni)
        check_gemm(Ch[r0:r1][mi, ni], ex, ab, True, "moe expert %d" % e)
    # the fused gather equals quantize-then-gather on sampled rows
    rows = np.linspace(0, len(src) - 1, 64).astype(np.int64)
    oq, os_ = oracle.quantize_act_rows(host_bits(X[torch.from_numpy(src[rows]).cuda()]))
    assert np.array_equal(hqx[rows], oq) and np.array_equal(hsx[:, rows], os_)


# ----------------------------------------------------------------- stream-K

@pytest.fixture(scope="module")
def workspace(f):
    return f.gemm_workspace()


def _flags_zero(f, ws):
    # the flag words (one per SM, first bytes of the workspace) are back to 0
    n = torch.cuda.get_device_properties(0).multi_processor_count
    return bool((ws[:4 * n] == 0).all())


@pytest.mark.parametrize("M,N,K,gran,out", [
    (256, 512, 8192, 128, torch.float32),     # 4 tiles, 64 K-blocks each: every tile split ~37 ways
    (1000, 1280, 4096, 128, torch.bfloat16),  # ragged rows, 40 tiles
    (384, 768, 2048, 1, torch.float32),       # per-column B scales
    (384, 768, 8192, 1, torch.bfloat16),      # per-column B scales split by stream-K (9 tiles, 576 K-blocks)
    (200, 384, 1024, 128, torch.bfloat16),    # N tail tile of 128 columns
])
def test_streamk_matches_oracle(f, workspace, M, N, K, gran, out):
    rng = np.random.default_rng(M + N + K + gran)
    Aq, Bq = rand_codes(rng, (M, K)), rand_codes(rng, (N, K))
    sA = rand_scales(rng, (K // 128, M))
    sB = rand_scales(rng, (N // 128, K // 128)) if gran == 128 else rand_scales(rng, (K // 128, N))
    dA, dsA, dB, dsB = dev(Aq), dev(sA), dev(Bq), dev(sB)
    C = f.gemm(dA, dsA, dB, dsB, out_dtype=out, sb_gran_n=gran, workspace=workspace)
    torch.cuda.synchronize()
    status_ok()
    assert _flags_zero(f, workspace)
    ex, ab, _ = oracle.gemm(Aq, sA, Bq, sB, sb_gran=gran)
    check_gemm(gemm_out_to_f64(C), ex, ab, out == torch.bfloat16, "stream-K %dx%dx%d" % (M, N, K))
    # deterministic: a second call gives the same bits
    C2 = f.gemm(dA, dsA, dB, dsB, out_dtype=out, sb_gran_n=gran, workspace=workspace)
    torch.cuda.synchronize()
    assert torch.equal(C.view(torch.int16) if out == torch.bfloat16 else C.view(torch.int32),
                       C2.view(torch.int16) if out == torch.bfloat16 else C2.view(torch.int32))


def test_streamk_wgrad_full_size(f, workspace):
    # Wgrad 2048x7168x8192: 448 tiles of 128x256 on the SMs (3.03 waves), the
    # case the balanced split is for
    dY, X = synth.wgrad_inputs(device="cuda")
    _, _, qdy, sdy = f.quantize_act(dY, row=False, col=True)
    _, _, qx, sx = f.quantize_act(X, row=False, col=True)
    C = f.gemm(qdy, sdy, qx, sx, out_dtype=torch.float32, sb_gran_n=1, workspace=workspace)
    C0 = f.gemm(qdy, sdy, qx, sx, out_dtype=torch.float32, sb_gran_n=1)
    torch.cuda.synchronize()
    status_ok()
    assert _flags_zero(f, workspace)
    mi, ni = sample_points(2048, 7168, seed=5)
    ex, ab, _ = oracle.gemm_points(to_np(qdy), to_np(sdy), to_np(qx), to_np(sx), mi, ni, sb_gran=1)
    check_gemm(gemm_out_to_f64(C)[mi, ni], ex, ab, False, "wgrad stream-K")
    # and it agrees with the data-parallel schedule to FP32 summation order
    d = (C - C0).abs().double().cpu().numpy()[mi, ni]
    assert (d <= 1e-5 * ab + 1e-30).all()


def test_workspace_too_small_is_rejected(f):
    A = torch.zeros(128, 128, dtype=torch.uint8, device="cuda")
    s = torch.ones(1, 128, dtype=torch.float32, device="cuda")
    sb = torch.ones(1, 1, dtype=torch.float32, device="cuda")
    C = torch.empty(128, 128, dtype=torch.float32, device="cuda")
    small = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(f.Fp8qError) as e:
        f.fp8q_gemm_ws(A, s, A, sb, C, 128, small)
    assert e.value.status == 8
