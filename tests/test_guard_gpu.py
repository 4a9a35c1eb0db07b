"""Out-of-bounds writes: every output of every entry point is placed between
guard regions filled with a canary byte, on shapes with ragged edges (row
tails, half N-tiles, stream-K splits, empty experts); after each call the
guards must be intact.  (compute-sanitizer is not available here; this is
the check that takes its place for writes.)"""
import numpy as np
import pytest
import torch

import synth
from helpers import status_ok

pytestmark = pytest.mark.gpu

GUARD = 4096
CANARY = 0xA5


class Guarded:
    """Device buffers carved out of one canary-filled allocation."""

    def __init__(self):
        self.parts = []

    def make(self, shape, dtype):
        nbytes = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        raw = torch.full((GUARD + ((nbytes + 15) // 16) * 16 + GUARD,), CANARY, dtype=torch.uint8, device="cuda")
        self.parts.append((raw, nbytes))
        return raw[GUARD:GUARD + nbytes].view(dtype).view(shape)

    def check(self, what):
        torch.cuda.synchronize()
        for raw, nbytes in self.parts:
            h = raw.cpu().numpy()
            assert np.all(h[:GUARD] == CANARY), what + ": write before an output"
            assert np.all(h[GUARD + nbytes:] == CANARY), what + ": write past an output"


def test_quantizers_stay_in_bounds():
    import fine_grained_fp8_quantize_b300 as f
    for dt in (torch.bfloat16, torch.float32):
        g = Guarded()
        x = synth.matrix(31, 1, 256, 384, 1.0, dtype=dt).cuda()
        qr, sr = g.make((256, 384), torch.uint8), g.make((3, 256), torch.float32)
        qc, sc = g.make((384, 256), torch.uint8), g.make((2, 384), torch.float32)
        f.fp8q_quantize_act(x, qr, sr, qc, sc)
        xr = synth.matrix(31, 2, 200, 384, 1.0, dtype=dt).cuda()  # ragged rows
        qr2, sr2 = g.make((200, 384), torch.uint8), g.make((3, 200), torch.float32)
        f.fp8q_quantize_act(xr, qr2, sr2)
        src = torch.tensor([5, 0, 199, 3, 77, 77, 1] * 11, dtype=torch.int32, device="cuda")
        qg, sg = g.make((77, 384), torch.uint8), g.make((3, 77), torch.float32)
        f.fp8q_quantize_act_gather(xr, src, qg, sg)
        w = synth.matrix(31, 3, 256, 384, 0.02, dtype=dt).cuda()
        qw, sw = g.make((256, 384), torch.uint8), g.make((2, 3), torch.float32)
        qt, st = g.make((384, 256), torch.uint8), g.make((3, 2), torch.float32)
        f.fp8q_quantize_weight_ex(w, qw, sw, qt, st)
        qm, sm = g.make((200, 384), torch.uint8), g.make((f.fp8q_mx_scale_bytes(200, 384),), torch.uint8)
        f.fp8q_mx_quantize(xr, qm, sm)
        status_ok()
        g.check("quantizers %s" % dt)


def rand_codes(shape, seed):
    rng = np.random.default_rng(seed)
    c = rng.integers(0, 256, shape).astype(np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x3F
    return torch.from_numpy(c).cuda()


def test_gemms_stay_in_bounds():
    import fine_grained_fp8_quantize_b300 as f
    g = Guarded()
    M, N, K = 200, 384, 256  # row tail and a half N-tile
    A, B = rand_codes((M, K), 1), rand_codes((N, K), 2)
    sA = torch.rand(K // 128, M, device="cuda") + 0.5
    sB = torch.rand(N // 128, K // 128, device="cuda") + 0.5
    for out in (torch.bfloat16, torch.float32):
        C = g.make((M, N), out)
        f.fp8q_gemm(A, sA, B, sB, C)
    sBc = torch.rand(K // 128, N, device="cuda") + 0.5
    Cw = g.make((M, N), torch.float32)
    f.fp8q_gemm_ex(A, sA, B, sBc, Cw, 1)
    # stream-K split: 448 tiles on the persistent grid
    Ms, Ns, Ks = 2048, 7168, 512
    As, Bs = rand_codes((Ms, Ks), 3), rand_codes((Ns, Ks), 4)
    sAs = torch.rand(Ks // 128, Ms, device="cuda") + 0.5
    sBs = torch.rand(Ks // 128, Ns, device="cuda") + 0.5
    Cs = g.make((Ms, Ns), torch.float32)
    ws = g.make((f.fp8q_gemm_workspace_size(),), torch.uint8)
    ws.zero_()
    f.fp8q_gemm_ws(As, sAs, Bs, sBs, Cs, 1, ws)
    # grouped: empty experts and ragged tails
    counts = [0, 70, 0, 129, 1, 0]
    off = torch.tensor(np.concatenate([[0], np.cumsum(counts)]).astype(np.int32), device="cuda")
    T = sum(counts)
    Ag = rand_codes((T, K), 5)
    sAg = torch.rand(K // 128, T, device="cuda") + 0.5
    Bg = rand_codes((len(counts), N, K), 6)
    sBg = torch.rand(len(counts), N // 128, K // 128, device="cuda") + 0.5
    Cg = g.make((T, N), torch.bfloat16)
    f.fp8q_grouped_gemm(Ag, sAg, Bg, sBg, Cg, off)
    # MX: row tail and a half N-tile
    sa8 = torch.full((f.fp8q_mx_scale_bytes(M, K),), 127, dtype=torch.uint8, device="cuda")
    sb8 = torch.full((f.fp8q_mx_scale_bytes(N, K),), 127, dtype=torch.uint8, device="cuda")
    Cm = g.make((M, N), torch.bfloat16)
    f.fp8q_mx_gemm(A, sa8, B, sb8, Cm)
    status_ok()
    g.check("gemms")
