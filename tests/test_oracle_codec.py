"""Pins of the oracle's E4M3 codec against things other than itself:
the format's definition worked by hand (golden file), a library decoder and
encoder (torch.float8_e4m3fn), and a brute-force nearest-value search."""
import os

import numpy as np
import pytest
import torch

import oracle
from conftest import GOLDEN

ALL = np.arange(256, dtype=np.uint8)


def torch_decode(codes):
    return torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(torch.float8_e4m3fn).float().numpy()


def _golden_values():
    rows = []
    with open(os.path.join(GOLDEN, "e4m3_notable_values.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            v, c = line.split()[:2]
            val = float.fromhex(v) if ("0x" in v and "p" in v) else float(v)
            rows.append((val, int(c, 16)))
    return rows


def test_golden_notable_values():
    rows = _golden_values()
    assert len(rows) >= 25
    vals = np.array([r[0] for r in rows], np.float32)
    want = np.array([r[1] for r in rows], np.uint8)
    got = oracle.e4m3_encode(vals)
    bad = [(float(v), hex(w), hex(g)) for v, w, g in zip(vals, want, got) if w != g]
    assert not bad, bad


def test_decode_matches_library_all_codes():
    mine = oracle.e4m3_decode(ALL)
    lib = torch_decode(ALL)
    nan = np.isnan(lib)
    assert np.array_equal(np.isnan(mine), nan)
    assert nan.sum() == 2                      # only 0x7F and 0xFF
    assert np.array_equal(mine[~nan], lib[~nan])
    # sign of zero
    assert np.signbit(mine[0x80]) and not np.signbit(mine[0x00])


def test_decode_grid_structure():
    v = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8)).astype(np.float64)
    assert v[0] == 0.0 and v[-1] == 448.0
    d = np.diff(v)
    assert (d > 0).all()                       # strictly increasing
    # spacing 2^-9 through the subnormals and the first normal binade, then
    # doubling every 8 codes
    for c in range(1, 0x7F):
        binade = 0 if c <= 16 else (c - 1) // 8 - 1
        assert d[c - 1] == 2.0 ** (-9 + binade), (c, d[c - 1])


def test_encode_roundtrip_all_codes():
    vals = oracle.e4m3_decode(ALL)
    ok = ~np.isnan(vals)
    enc = oracle.e4m3_encode(vals[ok])
    assert np.array_equal(enc, ALL[ok])


def test_midpoints_round_to_even():
    pos = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8)).astype(np.float64)
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    assert np.array_equal(mids.astype(np.float64), (pos[:-1] + pos[1:]) / 2)  # exact
    enc = oracle.e4m3_encode(mids)
    lo = np.arange(0, 0x7E)
    want = np.where(lo % 2 == 0, lo, lo + 1).astype(np.uint8)
    assert np.array_equal(enc, want)
    assert np.array_equal(oracle.e4m3_encode(-mids), want | 0x80)


def brute_force_encode(v):
    """Nearest E4M3 magnitude by exhaustive search (ties: even code),
    saturating to 448; sign copied."""
    mags = torch_decode(np.arange(0x7F, dtype=np.uint8)).astype(np.float64)
    out = np.empty(v.shape, np.uint8)
    for i, x in enumerate(v.astype(np.float64)):
        a = abs(x)
        if a >= 448.0:
            c = 0x7E
        else:
            dist = np.abs(mags - a)
            best = np.flatnonzero(dist == dist.min())
            c = best[0] if len(best) == 1 else [b for b in best if b % 2 == 0][0]
        out[i] = c | (0x80 if np.signbit(x) else 0)
    return out


def test_encode_vs_brute_force():
    rng = np.random.default_rng(1234)
    mag = 2.0 ** rng.uniform(-13, 10, 4000)
    sign = rng.choice([-1.0, 1.0], 4000)
    v = np.concatenate([(mag * sign), [0.0, -0.0, 448.0, 463.99, 464.0, 1e30, -1e-30]]).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(v), brute_force_encode(v))


def test_encode_vs_library_cast():
    # torch's float32 -> float8_e4m3fn cast rounds to nearest even but does
    # not saturate (values >= 464 go to NaN), so it pins |v| <= 464.
    rng = np.random.default_rng(99)
    v = (2.0 ** rng.uniform(-14, np.log2(464.0), 200000) * rng.choice([-1, 1], 200000)).astype(np.float32)
    v = v[np.abs(v) <= 464.0]
    lib = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(v), lib)


@pytest.mark.parametrize("x", [1e-45, 1e-40, 2.0 ** -126])
def test_encode_tiny_fp32(x):
    # fp32 subnormals and the smallest normal are far below 2^-10: they
    # round to zero with their sign
    assert oracle.e4m3_encode(np.array([x, -x], np.float32)).tolist() == [0x00, 0x80]
