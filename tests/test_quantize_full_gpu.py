"""Bit-exact parity of every quantizer mode at the full sizes of the five
workloads: every E4M3 code and every FP32 scale bit is compared with the
oracle, so the persistent kernels' later tiles (where each CTA's
double-buffered ring has wrapped many times) are checked byte for byte, not
only through the GEMM tolerance.

Groups: 1x128 activation tiles and 128x128 weight blocks -- dssusan.co.kr
page, the Figure 7 (a) passage; the 128x1 transposed copy that FP8 Wgrad
consumes -- "Is aI Hitting a Wall?", the Wgrad sentence.  E4M3 on all
tensors -- "Deepseek Ai News Expert Interview", the E4M3 passage.
Quantize-before-dispatch gather -- "Eliminate Deepseek Ai News For Good",
the dispatch passage."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import host_bits, status_ok, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def f():
    import fine_grained_fp8_quantize_b300 as f
    return f


def _eq(got, want, what):
    got, want = np.asarray(got), np.asarray(want)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    if got.dtype == np.float32:
        got, want = got.view(np.uint32), want.view(np.uint32)
    bad = got != want
    assert not bad.any(), "%s: %d mismatches, first at %s (gpu %r, oracle %r)" % (
        what, int(bad.sum()), tuple(np.argwhere(bad)[0]), got[bad][0], want[bad][0])


def _tiles_per_cta(f, tiles):
    # the persistent quantizers keep at most ~3 CTAs per SM: a full-size
    # launch gives each CTA many tiles, so its 2-deep ring wraps
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return tiles / (3 * sms)


def test_fprop_x_rows_full_size_4096x7168(f):
    # the Fprop activation, every row: X BF16 4096x7168 N(0,1), 0.1% x1e3
    X, _ = synth.fprop_inputs(device="cuda", N=128)
    q, s, _, _ = f.quantize_act(X, row=True, col=False)
    torch.cuda.synchronize()
    status_ok()
    oq, os_ = oracle.quantize_act_rows(host_bits(X))
    _eq(to_np(q), oq, "X codes")
    _eq(to_np(s), os_, "X scales")


def test_fprop_weight_full_size_18432x7168(f):
    # W BF16 18432x7168 N(0,0.02^2): 8064 blocks of 128x128, alone and with
    # the transposed copy (the Dgrad operand)
    _, W = synth.fprop_inputs(device="cuda", M=128)
    assert _tiles_per_cta(f, (18432 // 128) * (7168 // 128)) > 10
    oq, os_ = oracle.quantize_weight(host_bits(W))
    q, s = f.quantize_weight(W)
    torch.cuda.synchronize()
    status_ok()
    _eq(to_np(q), oq, "W codes")
    _eq(to_np(s), os_, "W scales")
    del q, s
    q, s, q_t, s_t = f.quantize_weight(W, transposed=True)
    torch.cuda.synchronize()
    status_ok()
    _eq(to_np(q), oq, "W codes (with transpose)")
    _eq(to_np(s), os_, "W scales (with transpose)")
    _eq(to_np(q_t), oq.T, "W^T codes")
    _eq(to_np(s_t), os_.T, "W^T scales")
    del q, s
    q_t2 = torch.empty(7168, 18432, dtype=torch.uint8, device="cuda")
    s_t2 = torch.empty(7168 // 128, 18432 // 128, dtype=torch.float32, device="cuda")
    f.fp8q_quantize_weight_ex(W, None, None, q_t2, s_t2)
    torch.cuda.synchronize()
    status_ok()
    _eq(to_np(q_t2), oq.T, "W^T codes (transpose only)")
    _eq(to_np(s_t2), os_.T, "W^T scales (transpose only)")


@pytest.mark.parametrize("which", ["dY", "X"])
def test_wgrad_operands_cols_only_full_size(f, which):
    # Wgrad operands: dY BF16 8192x2048 (N(0,1e-6), 0.5% x50) and X BF16
    # 8192x7168 (N(0,1)), each quantized only in 128x1 groups along tokens
    dY, X = synth.wgrad_inputs(device="cuda")
    T = dY if which == "dY" else X
    del dY, X
    _, _, q, s = f.quantize_act(T, row=False, col=True)
    torch.cuda.synchronize()
    status_ok()
    oq, os_ = oracle.quantize_act_cols(host_bits(T))
    _eq(to_np(q), oq, "%s^T codes" % which)
    _eq(to_np(s), os_, "%s^T scales" % which)


def test_moe_expert_weights_full_size(f):
    # every active expert's BF16 2048x7168 weight, quantized in one launch
    # over the stacked [E*N, K] tensor, then compared expert by expert
    off, _ = synth.moe_routing()
    counts = off[1:] - off[:-1]
    active = [int(e) for e in np.flatnonzero(counts)]
    E, N, K = 256, 2048, 7168
    _, W = synth.moe_inputs(device="cuda", experts=active)
    q, s = f.quantize_weight(W.view(E * N, K))
    torch.cuda.synchronize()
    status_ok()
    q = q.view(E, N, K)
    s = s.view(E, N // 128, K // 128)
    for e in active:
        oq, os_ = oracle.quantize_weight(host_bits(W[e]))
        _eq(to_np(q[e]), oq, "expert %d codes" % e)
        _eq(to_np(s[e]), os_, "expert %d scales" % e)
    # an expert nobody routes to has all-zero weights: codes 0, clamped scale
    idle = [e for e in range(E) if counts[e] == 0]
    if idle:
        e = idle[0]
        assert not bool(q[e].any())
        oq, os_ = oracle.quantize_weight(host_bits(W[e]))
        _eq(to_np(s[e]), os_, "idle expert %d scales" % e)


def test_moe_dispatch_gather_full_size(f):
    # quantize-before-dispatch: all 65,536 routed rows of the 8192x7168
    # tokens, gathered into expert order by the fused kernel
    off, src = synth.moe_routing()
    X = synth.matrix(4, 1, 8192, 7168, 1.0, device="cuda")
    q, s = f.quantize_act_gather(X, torch.from_numpy(src.astype(np.int32)).cuda())
    torch.cuda.synchronize()
    status_ok()
    oq, os_ = oracle.quantize_act_rows_gather(host_bits(X), src)
    _eq(to_np(q), oq, "gathered codes")
    _eq(to_np(s), os_, "gathered scales")


def test_dgrad_operand_rows_full_size_4096x18432(f):
    # the Dgrad left operand dY BF16 4096x18432, 1x128 rows over the 18432
    # output features (N(0,1e-6), 0.5% x50, as the Wgrad dY)
    dY = synth.matrix(5, 1, 4096, 18432, 1e-3, entry_frac=5e-3, entry_scale=50.0, device="cuda")
    q, s, _, _ = f.quantize_act(dY, row=True, col=False)
    torch.cuda.synchronize()
    status_ok()
    oq, os_ = oracle.quantize_act_rows(host_bits(dY))
    _eq(to_np(q), oq, "dY codes")
    _eq(to_np(s), os_, "dY scales")
