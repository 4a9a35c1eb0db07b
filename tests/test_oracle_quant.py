"""Pins of the oracle's quantizers (1x128 rows, 128x1 transposed copy,
128x128 weight blocks) against closed forms, invariants, a hand-worked
example and a library cast -- not against a retyping of its own formula.

Grouping: activations per 1x128 tile, weights per 128x128 block
(dssusan.co.kr page, the Figure 7 (a) passage); E4M3 on all tensors
("Deepseek Ai News Expert Interview", the E4M3/E5M2 passage)."""
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from conftest import GOLDEN


def bf16(a):
    """float array -> BF16 bits (uint16), round to nearest even via torch."""
    return synth.bf16_bits(torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16))


def from_bf16(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


def e4m3_ulp(v):
    """Spacing of the E4M3 grid at |v| (2^-9 below 2^-6)."""
    a = np.abs(v).astype(np.float64)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -6)))
    return 2.0 ** (e - 3)


def test_worked_example_golden():
    groups = {}
    cur = None
    with open(os.path.join(GOLDEN, "quant_worked_example.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            tok = line.split()
            if tok[0] == "group":
                cur = tok[1]
                groups[cur] = {"s": tok[2].split("=")[1], "el": []}
            else:
                groups[cur]["el"].append((int(tok[0]), tok[1], int(tok[3], 16)))
    assert set(groups) == {"A", "B", "C"}
    x = np.zeros((3, 128), np.float32)
    want = np.zeros((3, 128), np.uint8)
    for r, g in enumerate("ABC"):
        for j, v, c in groups[g]["el"]:
            x[r, j] = float.fromhex(v) if "0x" in v else float(v)
            want[r, j] = c
    xb = bf16(x)
    assert np.array_equal(from_bf16(xb), x)          # the example is exact in BF16
    q, s = oracle.quantize_act_rows(xb)
    assert np.array_equal(q, want), np.argwhere(q != want)
    assert s[0, 0] == np.float32(2.0 ** -7)
    assert s[0, 1] == np.float32(1.0)
    assert s[0, 2] == np.float32(np.float32(2.0 ** -100) / np.float32(448.0))


@pytest.mark.parametrize("j", [-20, -7, 0, 3])
def test_power_of_two_amax_reduces_to_plain_cast(j):
    # a group whose amax is 448 * 2^j has s = 2^j and inv = 2^-j exactly, so
    # its codes are the plain E4M3 cast (torch's) of x * 2^-j
    rng = np.random.default_rng(50 + j)
    x = (rng.standard_normal((256, 512)) * 40.0).astype(np.float32)
    x = from_bf16(bf16(x))
    x[:, ::128] = 448.0 * 2.0 ** j * np.sign(rng.standard_normal((256, 4)))  # one amax per group
    x = np.clip(x, -448.0 * 2.0 ** j, 448.0 * 2.0 ** j)
    xb = bf16(x)
    x = from_bf16(xb)
    q, s = oracle.quantize_act_rows(xb)
    assert (s == np.float32(2.0 ** j)).all()
    lib = torch.from_numpy(x * np.float32(2.0 ** -j)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q, lib)


def _check_groups(x, q, s, axis_groups):
    """Invariants of every group: the amax element maps to exactly +-448,
    no code exceeds 448, and dequantization error <= half an E4M3 ulp of
    x*inv times s (plus the few-ulp fp32 slack of x*inv and s*inv != 1)."""
    dq = oracle.e4m3_decode(q).astype(np.float64)
    for g_x, g_dq, g_s in axis_groups(x, dq, s):
        amax = np.abs(g_x).max()
        assert np.abs(g_dq).max() <= 448.0
        if amax > 2.0 ** -100:
            assert np.abs(g_dq).max() == 448.0
            v = g_x.astype(np.float64) * (448.0 / amax)
            bound = 0.5 * e4m3_ulp(v) * float(g_s) + 4 * 2.0 ** -24 * np.abs(g_x)
            assert (np.abs(g_dq * float(g_s) - g_x) <= bound).all()


def test_row_group_invariants():
    X = synth.matrix(11, 1, 256, 1024, 1.0, entry_frac=1e-2, entry_scale=1e3,
                     row_frac=0.05, row_scale=1e-3)
    xb = synth.bf16_bits(X)
    x = from_bf16(xb)
    q, s = oracle.quantize_act_rows(xb)

    def groups(x, dq, s):
        for m in range(x.shape[0]):
            for kb in range(x.shape[1] // 128):
                sl = slice(kb * 128, kb * 128 + 128)
                yield x[m, sl], dq[m, sl], s[kb, m]
    _check_groups(x, q, s, groups)


def test_col_group_invariants():
    X = synth.matrix(12, 1, 384, 256, 1.0, entry_frac=1e-2, entry_scale=1e3,
                     row_frac=0.05, row_scale=1e-3)
    xb = synth.bf16_bits(X)
    x = from_bf16(xb)
    qT, s = oracle.quantize_act_cols(xb)

    def groups(x, dqT, s):
        for k in range(x.shape[1]):
            for mb in range(x.shape[0] // 128):
                sl = slice(mb * 128, mb * 128 + 128)
                yield x[sl, k], dqT[k, sl], s[mb, k]
    _check_groups(x, qT, s, groups)


def test_weight_block_invariants():
    W = synth.matrix(13, 2, 384, 256, 0.02, entry_frac=1e-3, entry_scale=30.0)
    wb = synth.bf16_bits(W)
    w = from_bf16(wb)
    q, s = oracle.quantize_weight(wb)
    assert s.shape == (3, 2)

    def groups(w, dq, s):
        for nb in range(w.shape[0] // 128):
            for kb in range(w.shape[1] // 128):
                r = slice(nb * 128, nb * 128 + 128)
                c = slice(kb * 128, kb * 128 + 128)
                yield w[r, c].ravel(), dq[r, c].ravel(), s[nb, kb]
    _check_groups(w, q, s, groups)


def test_cols_equal_rows_of_transpose():
    # the 128x1 copy of X is the 1x128 quantization of X^T
    X = synth.matrix(14, 1, 256, 384, 1.0, entry_frac=1e-2, entry_scale=100.0)
    xb = synth.bf16_bits(X)
    qT, sc = oracle.quantize_act_cols(xb)
    qr, sr = oracle.quantize_act_rows(np.ascontiguousarray(xb.T))
    assert np.array_equal(qT, qr)
    assert np.array_equal(sc, sr)


def test_weight_equals_rows_when_block_amax_in_every_row():
    # if every row of a 128x128 block holds the block's amax, its 1x128 row
    # groups share the block's scale, so both quantizers agree
    rng = np.random.default_rng(3)
    w = rng.standard_normal((256, 384)).astype(np.float32) * 0.02
    for nb in range(2):
        for kb in range(3):
            amax = 0.1 * (1 + nb + 2 * kb)
            w[nb * 128:(nb + 1) * 128, kb * 128] = amax
    wb = bf16(w)
    qw, sw = oracle.quantize_weight(wb)
    qr, sr = oracle.quantize_act_rows(wb)
    assert np.array_equal(qw, qr)
    for nb in range(2):
        for kb in range(3):
            assert (sr[kb, nb * 128:(nb + 1) * 128] == sw[nb, kb]).all()


def test_zero_and_signed_zero_groups():
    x = np.zeros((2, 128), np.float32)
    x[1, :] = -0.0
    q, s = oracle.quantize_act_rows(bf16(x))
    assert (q[0] == 0x00).all() and (q[1] == 0x80).all()
    assert (s == np.float32(np.float32(2.0 ** -100) / np.float32(448.0))).all()


def test_fp32_input_equals_bf16_input_on_bf16_values():
    X = synth.matrix(15, 1, 128, 256, 1.0, entry_frac=1e-2, entry_scale=1e3)
    xb = synth.bf16_bits(X)
    a = oracle.quantize_act_rows(xb)
    b = oracle.quantize_act_rows(from_bf16(xb))
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    c = oracle.quantize_weight(xb)
    d = oracle.quantize_weight(from_bf16(xb))
    assert np.array_equal(c[0], d[0]) and np.array_equal(c[1], d[1])


def test_gather_equals_gather_of_quantized():
    # quantize-before-dispatch: 1x128 groups are row-local, so quantizing
    # gathered rows equals gathering quantized rows
    X = synth.matrix(16, 1, 64, 256, 1.0, entry_frac=1e-2, entry_scale=1e3)
    xb = synth.bf16_bits(X)
    src = np.array([5, 5, 0, 63, 17, 2, 2, 2, 40], np.int64)
    qg, sg = oracle.quantize_act_rows_gather(xb, src)
    q, s = oracle.quantize_act_rows(xb)
    assert np.array_equal(qg, q[src])
    assert np.array_equal(sg, s[:, src])
