"""Pins of the oracle's block-scaled GEMM:
  C = sum_kb sA[kb, m] * sB(kb, n) * P_kb[m, n],  P_kb = sum over 128 k of
  decode(Aq) * decode(Bq)
(promotion every 128 K with the scales applied there: "Eliminate Deepseek Ai
News For Good", the MMA-precision passage; inprokorea.com page, the
accumulation-interval passage; "Is aI Hitting a Wall?", the dequantization
passage).  Pinned by a brute-force per-element sum of dequantized products,
by torch's fp64 matmul, by the FP32 rounding-error bound of the pages'
promotion order, by exact scale linearity, and by the end-to-end error of
quantize-then-multiply against the unquantized product."""
import numpy as np
import pytest
import torch

import oracle
import synth


def rand_codes(rng, shape):
    c = rng.integers(0, 256, shape).astype(np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x3F            # no NaN codes
    return c


def rand_scales(rng, shape):
    return (2.0 ** rng.uniform(-12, 4, shape)).astype(np.float32)


def dequant_rows(q, s_kbm):
    """q[M,K] codes, s[K/128, M] scales -> fp64 A_dq[M,K] (per element)."""
    d = oracle.e4m3_decode(q).astype(np.float64)
    return d * np.repeat(s_kbm.T.astype(np.float64), 128, axis=1)


def dequant_b(q, sB, sb_gran):
    d = oracle.e4m3_decode(q).astype(np.float64)
    if sb_gran == 128:                               # sB[N/128, K/128]
        s = np.repeat(np.repeat(sB.astype(np.float64), 128, 0), 128, 1)
    else:                                            # sB[K/128, N]
        s = np.repeat(sB.T.astype(np.float64), 128, axis=1)
    return d * s


@pytest.mark.parametrize("sb_gran", [128, 1])
def test_brute_force_tiny(sb_gran):
    rng = np.random.default_rng(7 + sb_gran)
    M, N, K = 3, 130 if sb_gran == 1 else 256, 384
    Aq, Bq = rand_codes(rng, (M, K)), rand_codes(rng, (N, K))
    sA = rand_scales(rng, (K // 128, M))
    sB = rand_scales(rng, (N // 128, K // 128) if sb_gran == 128 else (K // 128, N))
    ex, ab, pg = oracle.gemm(Aq, sA, Bq, sB, sb_gran)
    da, db = oracle.e4m3_decode(Aq), oracle.e4m3_decode(Bq)
    for m in range(M):
        for n in range(N):
            tot = 0.0
            tabs = 0.0
            for k in range(K):
                a = float(da[m, k]) * float(sA[k // 128, m])
                if sb_gran == 128:
                    b = float(db[n, k]) * float(sB[n // 128, k // 128])
                else:
                    b = float(db[n, k]) * float(sB[k // 128, n])
                tot += a * b
                tabs += abs(a * b)
            assert abs(ex[m, n] - tot) <= 1e-12 * tabs
            assert abs(ab[m, n] - tabs) <= 1e-12 * tabs


@pytest.mark.parametrize("sb_gran", [128, 1])
def test_matches_library_matmul_fp64(sb_gran):
    rng = np.random.default_rng(21)
    M, N, K = 128, 256, 640
    Aq, Bq = rand_codes(rng, (M, K)), rand_codes(rng, (N, K))
    sA = rand_scales(rng, (K // 128, M))
    sB = rand_scales(rng, (N // 128, K // 128) if sb_gran == 128 else (K // 128, N))
    ex, ab, _ = oracle.gemm(Aq, sA, Bq, sB, sb_gran)
    A = torch.from_numpy(dequant_rows(Aq, sA))
    B = torch.from_numpy(dequant_b(Bq, sB, sb_gran))
    ref = (A @ B.T).numpy()
    absref = (A.abs() @ B.abs().T).numpy()
    assert np.allclose(ab, absref, rtol=1e-12, atol=0)
    assert (np.abs(ex - ref) <= 1e-12 * absref).all()


def test_pages_order_within_fp32_bound():
    # acc = fl32(acc + fl32(fl32(P)*fl32(sA*sB))): KB roundings of the sum,
    # one each of P, sA*sB and the product -> |pages - exact| <=
    # (KB + 3) * 2^-24 * sum|a b| (first order)
    rng = np.random.default_rng(8)
    M, N, K = 64, 128, 2048
    Aq, Bq = rand_codes(rng, (M, K)), rand_codes(rng, (N, K))
    sA = rand_scales(rng, (K // 128, M))
    sB = rand_scales(rng, (N // 128, K // 128))
    ex, ab, pg = oracle.gemm(Aq, sA, Bq, sB, 128)
    KB = K // 128
    err = np.abs(pg.astype(np.float64) - ex)
    assert (err <= (KB + 3) * 2.0 ** -24 * ab * 1.01).all()
    assert err.max() > 0                             # the fl32 order does round


def test_scale_linearity_exact():
    rng = np.random.default_rng(9)
    M, N, K = 16, 128, 512
    Aq, Bq = rand_codes(rng, (M, K)), rand_codes(rng, (N, K))
    sA = rand_scales(rng, (K // 128, M))
    sB = rand_scales(rng, (N // 128, K // 128))
    ex, _, pg = oracle.gemm(Aq, sA, Bq, sB)
    ex2, _, pg2 = oracle.gemm(Aq, sA * np.float32(4.0), Bq, sB * np.float32(0.5))
    assert np.array_equal(ex2, 2.0 * ex) and np.array_equal(pg2, np.float32(2.0) * pg)
    # a single K-block's scale only moves that block's term
    sA3 = sA.copy()
    sA3[1, :] = 0.0
    ex3, _, _ = oracle.gemm(Aq, sA3, Bq, sB)
    sA4 = np.zeros_like(sA)
    sA4[1, :] = sA[1, :]
    ex4, _, _ = oracle.gemm(Aq, sA4, Bq, sB)
    assert np.allclose(ex3 + ex4, ex, rtol=1e-13, atol=1e-300)


def test_points_equal_full():
    rng = np.random.default_rng(10)
    M, N, K = 40, 256, 384
    Aq, Bq = rand_codes(rng, (M, K)), rand_codes(rng, (N, K))
    sA = rand_scales(rng, (K // 128, M))
    sB = rand_scales(rng, (N // 128, K // 128))
    ex, ab, pg = oracle.gemm(Aq, sA, Bq, sB)
    mi = rng.integers(0, M, 500)
    ni = rng.integers(0, N, 500)
    pe, pa, pp = oracle.gemm_points(Aq, sA, Bq, sB, mi, ni)
    assert np.array_equal(pe, ex[mi, ni]) and np.array_equal(pa, ab[mi, ni])
    assert np.array_equal(pp, pg[mi, ni])


def test_grouped_equals_dense_slices():
    rng = np.random.default_rng(11)
    E, N, K = 5, 256, 256
    counts = np.array([0, 130, 1, 0, 77])             # empty experts and ragged M
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    T = int(off[-1])
    Aq = rand_codes(rng, (T, K))
    sA = rand_scales(rng, (K // 128, T))
    Bq = rand_codes(rng, (E, N, K))
    sB = rand_scales(rng, (E, N // 128, K // 128))
    mi = np.repeat(np.arange(T), N)
    ni = np.tile(np.arange(N), T)
    ge, ga, gp = oracle.grouped_gemm_points(Aq, sA, Bq, sB, off, mi, ni)
    ge = ge.reshape(T, N)
    for e in range(E):
        r0, r1 = off[e], off[e + 1]
        if r1 == r0:
            continue
        de, _, _ = oracle.gemm(Aq[r0:r1], np.ascontiguousarray(sA[:, r0:r1]), Bq[e], sB[e])
        assert np.array_equal(ge[r0:r1], de)


def test_config1_quantize_then_gemm_approximates_product():
    # Tiny end-to-end case (seed 0): A BF16 128x512 N(0,1) with 1% x100,
    # B BF16 512x128 N(0, 0.02^2).  Dequantized codes carry a relative error
    # of at most 2^-4 per element (half an E4M3 ulp), so
    # |C_fp8 - A.B| <= (2 * 2^-4 + 2^-8) * sum|a||b|.  This pins the scale
    # convention (s multiplies codes back) and the operand layouts.
    A, Bt = synth.tiny_gemm_inputs(seed=0)
    qa, sa = oracle.quantize_act_rows(synth.bf16_bits(A))
    qb, sb = oracle.quantize_weight(synth.bf16_bits(Bt))
    ex, ab, pg = oracle.gemm(qa, sa, qb, sb)
    Af = A.double()
    Bf = Bt.double()
    ref = (Af @ Bf.T).numpy()
    absref = (Af.abs() @ Bf.abs().T).numpy()
    err = np.abs(ex - ref)
    assert (err <= (2 * 2.0 ** -4 + 2.0 ** -8) * absref).all()
    # and it is a real approximation, not a loose bound met by chance
    assert np.median(err / absref) < 0.02
