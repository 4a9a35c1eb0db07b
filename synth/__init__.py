"""Seeded synthetic inputs for the FP8 quantization / GEMM workloads.

This module serves both the CUDA path (tests, bench) and the CPU oracle.  It
holds none of the method's arithmetic: it only draws the input tensors and
the MoE routing that shapes the grouped workload.

Generator: SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014) evaluated at a counter, so any element can
be drawn independently on any device:

    z = base(seed, stream) + (i + 1) * 0x9E3779B97F4A7C15      (mod 2^64)
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9
    z = (z ^ (z >> 27)) * 0x94D049BB133111EB
    out = z ^ (z >> 31)

Uniforms take the top 24 bits, u = (out >> 40 + 0.5) / 2^24, in (0, 1).
Normals use Box-Muller on two independent streams.  Values are formed in
FP32 and rounded to BF16 (round to nearest even) by the dtype cast.
Torch integer arithmetic wraps modulo 2^64 on CPU and CUDA; right shifts are
made logical by masking.
"""
import math

import numpy as np
import torch

_GAMMA = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB
_CHUNK = 1 << 25


def _s64(u):
    """uint64 constant -> the int64 with the same bits."""
    u &= (1 << 64) - 1
    return u - (1 << 64) if u >= (1 << 63) else u


def _srl(z, s):
    """Logical right shift of int64 tensor z by s bits."""
    return (z >> s) & ((1 << (64 - s)) - 1)


def _mix(z):
    z = (z ^ _srl(z, 30)) * _s64(_M1)
    z = (z ^ _srl(z, 27)) * _s64(_M2)
    return z ^ _srl(z, 31)


def _mix_int(x):
    """Python-int SplitMix64 output function (for stream bases)."""
    m = (1 << 64) - 1
    x = (x + _GAMMA) & m
    x = ((x ^ (x >> 30)) * _M1) & m
    x = ((x ^ (x >> 27)) * _M2) & m
    return x ^ (x >> 31)


def stream_base(seed, stream):
    return _s64(_mix_int(_mix_int(int(seed)) ^ (int(stream) * 0xD1B54A32D192ED03)))


def uniform(seed, stream, n, device="cpu", start=0):
    """n uniforms in (0, 1) as float32 for counters start .. start+n-1."""
    base = stream_base(seed, stream)
    out = torch.empty(n, dtype=torch.float32, device=device)
    for c0 in range(0, n, _CHUNK):
        c1 = min(n, c0 + _CHUNK)
        i = torch.arange(start + c0 + 1, start + c1 + 1, dtype=torch.int64, device=device)
        z = _mix(i * _s64(_GAMMA) + base)
        top = _srl(z, 40).to(torch.float32)
        out[c0:c1] = (top + 0.5) * (1.0 / 16777216.0)
    return out


def _normal_range(seed, stream, c0, c1, std, device):
    """N(0, std^2) draws for counters c0 .. c1-1 of one normal stream."""
    u1 = uniform(seed, 2 * stream, c1 - c0, device, start=c0)
    u2 = uniform(seed, 2 * stream + 1, c1 - c0, device, start=c0)
    return torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * math.pi) * u2) * std


def normal(seed, stream, n, std=1.0, device="cpu"):
    """n N(0, std^2) float32 draws (Box-Muller over two uniform streams)."""
    out = torch.empty(n, dtype=torch.float32, device=device)
    for c0 in range(0, n, _CHUNK):
        c1 = min(n, c0 + _CHUNK)
        out[c0:c1] = _normal_range(seed, stream, c0, c1, std, device)
    return out


def matrix(seed, stream, rows, cols, std=1.0, entry_frac=0.0, entry_scale=1.0,
           row_frac=0.0, row_scale=1.0, dtype=torch.bfloat16, device="cpu"):
    """A [rows, cols] matrix of N(0, std^2) entries with optional outliers.

    entry_frac of the entries (chosen by an independent uniform < entry_frac)
    are multiplied by entry_scale; row_frac of the rows by row_scale.  Built
    in FP32, then cast to ``dtype`` (BF16: round to nearest even)."""
    n = rows * cols
    out = torch.empty(n, dtype=dtype, device=device)
    rmask = None
    if row_frac > 0.0:
        rmask = uniform(seed, 100 * stream + 3, rows, device) < row_frac
    for c0 in range(0, n, _CHUNK):
        c1 = min(n, c0 + _CHUNK)
        v = _normal_range(seed, 100 * stream, c0, c1, std, device)
        if entry_frac > 0.0:
            u = uniform(seed, 100 * stream + 2, c1 - c0, device, start=c0)
            v = torch.where(u < entry_frac, v * entry_scale, v)
        if rmask is not None:
            r = torch.arange(c0, c1, device=device) // cols
            v = torch.where(rmask[r], v * row_scale, v)
        out[c0:c1] = v.to(dtype)
    return out.view(rows, cols)


def bf16_bits(t):
    """Host numpy uint16 view of a BF16 tensor's bits (oracle input form)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


# --------------------------------------------------------------------------
# The five workloads (shapes and value recipes; seeds 0..4).
# --------------------------------------------------------------------------

def tiny_gemm_inputs(device="cpu", seed=0):
    """A BF16 128x512 N(0,1) with 1% of entries x100; B BF16 512x128
    N(0, 0.02^2), returned as its transpose Bt[128, 512] (K contiguous)."""
    A = matrix(seed, 1, 128, 512, 1.0, entry_frac=0.01, entry_scale=100.0, device=device)
    B = matrix(seed, 2, 512, 128, 0.02, device=device)
    return A, B.t().contiguous()


def act_quant_inputs(device="cpu", seed=1, T=16384, H=7168):
    """X BF16 [T, H] N(0,1); 0.1% of entries x1e3; 1% of rows x1e-3."""
    return matrix(seed, 1, T, H, 1.0, entry_frac=1e-3, entry_scale=1e3,
                  row_frac=0.01, row_scale=1e-3, device=device)


def fprop_inputs(device="cpu", seed=2, M=4096, N=18432, K=7168):
    """X BF16 [M, K] N(0,1) with 0.1% entries x1e3; W BF16 [N, K] N(0, 0.02^2)
    (PyTorch Linear layout of the K->N projection)."""
    X = matrix(seed, 1, M, K, 1.0, entry_frac=1e-3, entry_scale=1e3, device=device)
    W = matrix(seed, 2, N, K, 0.02, device=device)
    return X, W


def wgrad_inputs(device="cpu", seed=3, T=8192, Dout=2048, Din=7168):
    """dY BF16 [T, Dout] N(0, 1e-6) with 0.5% entries x50; X BF16 [T, Din] N(0,1)."""
    dY = matrix(seed, 1, T, Dout, 1e-3, entry_frac=5e-3, entry_scale=50.0, device=device)
    X = matrix(seed, 2, T, Din, 1.0, device=device)
    return dY, X


def moe_routing(seed=4, T=8192, E=256, topk=8):
    """Top-k expert choice per token by sigmoid(logit) + bias with logits
    N(0,1) [T, E] and bias N(0, 0.5^2) [E] (skewed loads).  Ties go to the
    lower expert index.  Returns (row_offsets int64[E+1], src_token int64[T*topk])
    with rows grouped by expert, tokens ascending inside an expert."""
    logits = normal(seed, 7, T * E).view(T, E).numpy().astype(np.float32)
    bias = normal(seed, 8, E, std=0.5).numpy().astype(np.float32)
    score = (1.0 / (1.0 + np.exp(-logits))).astype(np.float32) + bias[None, :]
    order = np.argsort(-score, axis=1, kind="stable")[:, :topk]
    tok = np.repeat(np.arange(T, dtype=np.int64), topk)
    exp = order.reshape(-1).astype(np.int64)
    perm = np.lexsort((tok, exp))
    counts = np.bincount(exp, minlength=E)
    offsets = np.zeros(E + 1, np.int64)
    offsets[1:] = np.cumsum(counts)
    return offsets, tok[perm]


def moe_inputs(device="cpu", seed=4, T=8192, H=7168, E=256, N=2048, experts=None):
    """Tokens BF16 [T, H] N(0,1); expert weights BF16 [E, N, H] N(0, 0.02^2).
    ``experts`` limits which experts' weights are drawn (others left zero)."""
    X = matrix(seed, 1, T, H, 1.0, device=device)
    W = torch.zeros(E, N, H, dtype=torch.bfloat16, device=device)
    for e in (range(E) if experts is None else experts):
        W[e] = matrix(seed, 1000 + e, N, H, 0.02, device=device)
    return X, W
