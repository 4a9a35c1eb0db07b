"""Pins of the oracle's MX variant (1x32 groups, power-of-two E8M0 scales):
the shared exponent against the float's own bit pattern, the E8M0 byte
against torch's float8_e8m0fnu cast, the element codes against torch's
float8_e4m3fn cast, closed-form round trips, and the GEMM against exact
rational arithmetic and an fp64 library matmul.

The pages only say that the fine-grained strategy follows the microscaling
formats and that Blackwell tensor cores support them ("Deepseek Ai News
Expert Interview", the DualPipe / microscaling paragraph); the conversion
pinned here is the one the MX formats define: shared exponent
floor(log2(amax)) - 8, clamped to [-127, 127], elements E4M3(x / 2^e)."""
from fractions import Fraction

import numpy as np
import torch

import oracle
import synth


def floor_log2_bits(a):
    """floor(log2(a)) of a positive float32 from its bit pattern (normal
    numbers: biased exponent - 127; subnormals: position of the top set
    mantissa bit - 149)."""
    bits = int(np.float32(a).view(np.uint32)) & 0x7FFFFFFF
    e = bits >> 23
    if e:
        return e - 127
    return (bits.bit_length() - 1) - 149


def expected_shared_exp(a):
    if a == 0:
        return -127
    return max(-127, min(127, floor_log2_bits(a) - 8))


def test_shared_exp_against_bit_pattern():
    rng = np.random.default_rng(11)
    vals = [0.0, 1.0, 448.0, 255.99, 256.0, 0.5, 2.0 ** -126, 2.0 ** -133, 2.0 ** -149, 3.0e38,
            np.nextafter(np.float32(2.0), np.float32(0)), np.float32(2.0 ** -118), np.float32(2.0 ** -119),
            np.float32(2.0 ** -120)]
    vals += list((10.0 ** rng.uniform(-44, 38, 4000)).astype(np.float32))
    vals += [np.float32(2.0 ** k) for k in range(-149, 128)]
    for a in vals:
        a = float(np.float32(a))
        assert oracle.mx_shared_exp(a) == expected_shared_exp(a), a


def test_e8m0_byte_matches_torch():
    x = synth.matrix(5, 1, 64, 256, 1.0, entry_frac=0.02, entry_scale=1e4, row_frac=0.1, row_scale=1e-20)
    _, e8 = oracle.mx_quantize_rows(synth.bf16_bits(x))
    xf = x.float().numpy()
    amax = np.abs(xf).reshape(64, 8, 32).max(axis=2)
    for r in range(64):
        for g in range(8):
            se = expected_shared_exp(float(amax[r, g]))
            code = int(torch.tensor([2.0 ** se], dtype=torch.float64).to(torch.float8_e8m0fnu)
                       .view(torch.uint8).item())
            assert int(e8[r, g]) == code


def test_codes_match_torch_cast():
    """Within the E4M3 range torch's RNE cast decides each code; above it the
    MX conversion saturates to +-448 (0x7E / 0xFE)."""
    x = synth.matrix(6, 1, 96, 512, 1.0, entry_frac=0.01, entry_scale=300.0)
    q, e8 = oracle.mx_quantize_rows(synth.bf16_bits(x))
    xf = x.float().numpy()
    inv = np.ldexp(np.float32(1.0), -(e8.astype(np.int32) - 127)).astype(np.float32)
    v = (xf.reshape(96, 16, 32) * inv[:, :, None]).reshape(96, 512).astype(np.float32)
    t = torch.from_numpy(np.clip(v, -448.0, 448.0)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    big = np.abs(v) >= 464.0
    exp = np.where(big, np.where(v < 0, 0xFE, 0x7E), t).astype(np.uint8)
    assert np.array_equal(q, exp)
    # some groups really do saturate (x / X reaches 511.x)
    assert np.any(np.abs(v) > 448.0)


def test_group_invariants():
    x = synth.matrix(7, 1, 128, 1024, 1.0, entry_frac=0.001, entry_scale=1e3, row_frac=0.05, row_scale=1e-3)
    q, e8 = oracle.mx_quantize_rows(synth.bf16_bits(x))
    d = torch.from_numpy(q).view(torch.float8_e4m3fn).to(torch.float64).numpy().reshape(128, 32, 32)
    gmax = np.abs(d).max(axis=2)
    assert np.all(gmax >= 256.0) and np.all(gmax <= 448.0)
    # dequantization error: half an E4M3 ulp of x / X, or the saturation gap
    xf = x.double().numpy().reshape(128, 32, 32)
    X = np.ldexp(1.0, e8.astype(np.int64) - 127)[:, :, None]
    v = xf / X
    a = np.abs(v)
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(a, 2.0 ** -6))) - 3)
    err = np.abs(d - v)
    assert np.all((err <= 0.5 * ulp) | ((a > 448.0) & (np.abs(d) == 448.0)))


def test_closed_form_round_trip():
    """Groups built as E4M3 values times 2^t, with a largest element in
    [256, 448], come back as the same codes with shared exponent t."""
    rng = np.random.default_rng(3)
    rows, G = 16, 8
    codes = rng.integers(0, 0x7F, size=(rows, G * 32)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x10          # no NaN patterns
    codes[:, ::32] = rng.integers(0x78, 0x7F, size=(rows, G)).astype(np.uint8)  # one element in [256, 448] per group
    codes |= (rng.integers(0, 2, size=codes.shape).astype(np.uint8) << 7)
    t = rng.integers(-100, 100, size=(rows, G))
    dec = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    x = (dec.reshape(rows, G, 32) * np.ldexp(1.0, t)[:, :, None]).reshape(rows, G * 32).astype(np.float32)
    q, e8 = oracle.mx_quantize_rows(x)
    assert np.array_equal(e8.astype(np.int64) - 127, t)
    assert np.array_equal(q, codes)


def test_all_zero_group_and_tiny_group():
    x = np.zeros((2, 64), np.float32)
    x[1, 32:] = np.float32(2.0 ** -140)     # subnormal FP32: shared exponent clamps to -127
    q, e8 = oracle.mx_quantize_rows(x)
    assert list(e8[0]) == [0, 0] and list(e8[1]) == [0, 0]
    assert np.all(q[0] == 0) and np.all(q[1, :32] == 0)
    # 2^-140 / 2^-127 = 2^-13 is below half the smallest E4M3 subnormal (2^-10): zero
    assert np.all(q[1, 32:] == 0)


def _decode(c):
    return torch.from_numpy(np.ascontiguousarray(c)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_gemm_bruteforce_fractions():
    rng = np.random.default_rng(5)
    M, N, K = 3, 4, 96
    Aq = rng.integers(0, 256, size=(M, K)).astype(np.uint8)
    Bq = rng.integers(0, 256, size=(N, K)).astype(np.uint8)
    Aq[(Aq & 0x7F) == 0x7F] = 0x01
    Bq[(Bq & 0x7F) == 0x7F] = 0x02
    ea = rng.integers(100, 150, size=(M, K // 32)).astype(np.uint8)
    eb = rng.integers(100, 150, size=(N, K // 32)).astype(np.uint8)
    da, db = _decode(Aq), _decode(Bq)
    mi, ni = np.repeat(np.arange(M), N), np.tile(np.arange(N), M)
    ex, ab = oracle.mx_gemm_points(Aq, ea, Bq, eb, mi, ni)
    for i, (m, n) in enumerate(zip(mi, ni)):
        s = Fraction(0)
        sa = Fraction(0)
        for k in range(K):
            g = k // 32
            sc = Fraction(2) ** (int(ea[m, g]) - 127 + int(eb[n, g]) - 127)
            p = Fraction(float(da[m, k])) * Fraction(float(db[n, k])) * sc
            s += p
            sa += abs(p)
        assert abs(Fraction(ex[i]) - s) <= sa * Fraction(1, 2 ** 50)
        assert abs(Fraction(ab[i]) - sa) <= sa * Fraction(1, 2 ** 50)


def test_gemm_matches_fp64_matmul():
    x = synth.matrix(8, 1, 128, 512, 1.0, entry_frac=0.01, entry_scale=100.0)
    w = synth.matrix(8, 2, 256, 512, 0.02)
    qa, ea = oracle.mx_quantize_rows(synth.bf16_bits(x))
    qb, eb = oracle.mx_quantize_rows(synth.bf16_bits(w))
    A = torch.from_numpy(_decode(qa) * np.repeat(np.ldexp(1.0, ea.astype(np.int64) - 127), 32, axis=1))
    B = torch.from_numpy(_decode(qb) * np.repeat(np.ldexp(1.0, eb.astype(np.int64) - 127), 32, axis=1))
    ref = (A @ B.T).numpy()
    mi, ni = np.repeat(np.arange(128), 256), np.tile(np.arange(256), 128)
    ex, ab = oracle.mx_gemm_points(qa, ea, qb, eb, mi, ni)
    assert np.all(np.abs(ex - ref.reshape(-1)) <= 1e-13 * ab + 1e-300)
    # and it approximates the unquantized product: each element is off by at
    # most 1/16 of itself (RNE, 3 mantissa bits) or 1/8 when it saturates
    # (511.x -> 448), so each product by at most (1 + 1/8)^2 - 1 of itself
    full = (x.double() @ w.double().T).numpy().reshape(-1)
    assert np.max(np.abs(ex - full) / (ab + 1e-30)) < 0.266
    assert np.median(np.abs(ex - full) / (ab + 1e-30)) < 0.02
