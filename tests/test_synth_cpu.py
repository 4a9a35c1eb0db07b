"""The seeded input generator (`synth/`): SplitMix64 against its published
reference outputs, determinism, the value recipes (outlier fractions, row
scaling, BF16 rounding) and the MoE routing invariants.  No GPU needed."""
import numpy as np
import torch

import synth


def test_splitmix64_reference_outputs():
    # SplitMix64 (Steele, Lea & Flood 2014) from state 0: the first outputs of
    # the reference implementation
    want = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    assert synth._mix_int(0) == want[0]
    i = torch.arange(1, 4, dtype=torch.int64)
    z = synth._mix(i * synth._s64(synth._GAMMA))
    got = [int(v) & ((1 << 64) - 1) for v in z.tolist()]
    assert got == want


def test_draws_are_deterministic_and_streams_differ():
    a = synth.matrix(3, 1, 64, 256, 1.0)
    b = synth.matrix(3, 1, 64, 256, 1.0)
    c = synth.matrix(3, 2, 64, 256, 1.0)
    d = synth.matrix(4, 1, 64, 256, 1.0)
    assert torch.equal(a, b)
    assert not torch.equal(a, c) and not torch.equal(a, d)
    # counters: a chunk drawn from an offset equals the tail of a longer draw
    u = synth.uniform(9, 5, 1000)
    v = synth.uniform(9, 5, 400, start=600)
    assert torch.equal(u[600:], v)


def test_uniform_and_normal_moments():
    u = synth.uniform(1, 1, 1 << 20).double()
    assert 0.0 < float(u.min()) and float(u.max()) < 1.0
    assert abs(float(u.mean()) - 0.5) < 2e-3 and abs(float(u.var()) - 1.0 / 12.0) < 2e-3
    x = synth.normal(1, 2, 1 << 20, std=2.0).double()
    assert abs(float(x.mean())) < 1e-2 and abs(float(x.std()) - 2.0) < 1e-2


def test_outlier_and_row_recipes():
    x = synth.matrix(5, 3, 512, 1024, 1.0, entry_frac=0.01, entry_scale=1e3, row_frac=0.1, row_scale=1e-3,
                     dtype=torch.float32)
    big = (x.abs() > 20.0).double().mean()
    assert 0.007 < float(big) < 0.013           # ~1% of entries scaled by 1e3 (a few are tiny rows)
    y = synth.matrix(5, 4, 2048, 256, 1.0, row_frac=0.1, row_scale=1e-3, dtype=torch.float32)
    small_rows = (y.abs().amax(dim=1) < 0.05).double().mean()
    assert 0.08 < float(small_rows) < 0.12      # ~10% of rows scaled by 1e-3
    # the BF16 form is the round-to-nearest-even cast of the FP32 values
    xb = synth.matrix(5, 3, 512, 1024, 1.0, entry_frac=0.01, entry_scale=1e3, row_frac=0.1, row_scale=1e-3)
    assert xb.dtype == torch.bfloat16 and torch.equal(xb, x.to(torch.bfloat16))


def test_moe_routing_invariants():
    T, E, k = 512, 64, 8
    off, src = synth.moe_routing(seed=4, T=T, E=E, topk=k)
    assert off[0] == 0 and off[-1] == T * k and np.all(np.diff(off) >= 0)
    assert np.array_equal(np.bincount(src, minlength=T), np.full(T, k))  # every token k times
    for e in range(E):
        seg = src[off[e]:off[e + 1]]
        assert np.all(np.diff(seg) > 0)  # tokens ascending, no token twice per expert
    # brute force: token t goes to the k best-scoring experts, ties to the lower index
    logits = synth.normal(4, 7, T * E).view(T, E).numpy().astype(np.float32)
    bias = synth.normal(4, 8, E, std=0.5).numpy().astype(np.float32)
    score = (1.0 / (1.0 + np.exp(-logits))).astype(np.float32) + bias[None, :]
    chosen = {e: set(src[off[e]:off[e + 1]].tolist()) for e in range(E)}
    for t in range(0, T, 37):
        best = sorted(range(E), key=lambda e: (-float(score[t, e]), e))[:k]
        assert all(t in chosen[e] for e in best)
