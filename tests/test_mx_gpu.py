"""GPU parity of the MX variant through the C ABI: the 1x32 quantizer
(codes and E8M0 scale bytes bit-exact with the oracle) and the GEMM whose
tensor cores apply the power-of-two scales (within the GEMM tolerance of the
oracle's exact result).

The pages tie the fine-grained strategy to the microscaling formats that
Blackwell tensor cores support ("Deepseek Ai News Expert Interview", the
DualPipe / microscaling paragraph); the oracle states the MX conversion.

The oracle keeps scales row-major (e8[rows][K/32]); the library keeps them in
the tiled layout of include/fp8q.h.  `tile_scales` below is that layout's
index map, written from the header's definition."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import check_gemm, gemm_out_to_f64, sample_points, status_ok, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def f():
    import fine_grained_fp8_quantize_b300 as f
    return f


def tile_scales(e8, rows, K):
    """Row-major e8[rows][K/32] -> the library's tiled bytes
    s[K/128][ceil(rows/128)][512], byte (r%32)*16 + (r/32)*4 + c of the chunk
    of row tile r/128 and K-block g/4 (c = g%4); padding rows hold 127."""
    RT, KT = (rows + 127) // 128, K // 128
    out = np.full((KT, RT, 512), 127, np.uint8)
    r = np.arange(rows)[:, None]
    g = np.arange(K // 32)[None, :]
    rr = r % 128
    out[g // 4, r // 128, (rr % 32) * 16 + (rr // 32) * 4 + g % 4] = e8[:rows]
    return out.reshape(-1)


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def rand_codes(rng, shape):
    c = rng.integers(0, 256, shape).astype(np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x3F
    return c


def run_quant(f, x):
    rows, K = x.shape
    q = torch.empty(rows, K, dtype=torch.uint8, device="cuda")
    s = torch.full((f.fp8q_mx_scale_bytes(rows, K),), 0xEE, dtype=torch.uint8, device="cuda")
    f.fp8q_mx_quantize(x, q, s)
    status_ok()
    return to_np(q), to_np(s)


def oracle_input(x):
    return synth.bf16_bits(x) if x.dtype == torch.bfloat16 else to_np(x)


@pytest.mark.parametrize("rows,K,dtype", [(384, 512, torch.bfloat16), (200, 384, torch.bfloat16),
                                          (256, 256, torch.float32), (1, 128, torch.bfloat16),
                                          (129, 1024, torch.float32)])
def test_quantize_bit_exact(f, rows, K, dtype):
    x = synth.matrix(21, 1, rows, K, 1.0, entry_frac=0.01, entry_scale=1e3, row_frac=0.1, row_scale=1e-3,
                     dtype=dtype).cuda()
    q, s = run_quant(f, x)
    oq, oe = oracle.mx_quantize_rows(oracle_input(x.cpu()))
    assert np.array_equal(q, oq)
    assert np.array_equal(s, tile_scales(oe, rows, K))


def test_quantize_extreme_values(f):
    """Zero groups, FP32 subnormals, the largest floats, exact powers of two
    and values on E4M3 rounding ties."""
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((256, 512)) * 10.0 ** rng.integers(-30, 30, (256, 1))).astype(np.float32)
    x[0, :64] = 0.0
    x[1, :32] = np.float32(2.0 ** -140)
    x[1, 32:64] = -np.float32(2.0 ** -149)
    x[2, :32] = np.float32(3.0e38)
    x[3, :32] = np.float32(2.0) ** np.arange(-16, 16)
    x[4, :32] = (np.arange(32) + 0.5).astype(np.float32) * np.float32(2.0 ** -3)   # ties at small codes
    x[5, :32] = -0.0
    xt = torch.from_numpy(x).cuda()
    q, s = run_quant(f, xt)
    oq, oe = oracle.mx_quantize_rows(x)
    assert np.array_equal(q, oq)
    assert np.array_equal(s, tile_scales(oe, 256, 512))


def test_quantize_full_size_act_16384x7168(f):
    """The 16384x7168 activation at full size, checked on sampled rows (the
    quantization is row-local): one row per 128-row tile plus the last."""
    X = synth.act_quant_inputs(device="cuda")
    rows, K = X.shape
    q, s = run_quant(f, X)
    rng = np.random.default_rng(9)
    pick = np.array(sorted({int(t * 128 + rng.integers(0, 128)) for t in range(rows // 128)} | {rows - 1}))
    oq, oe = oracle.mx_quantize_rows(synth.bf16_bits(X[torch.from_numpy(pick).cuda()]))
    assert np.array_equal(q[pick], oq)
    assert np.array_equal(untile(s.reshape(K // 128, rows // 128, 512), pick, K), oe)


def run_gemm(f, Aq, ea, Bq, eb, out):
    M, K = Aq.shape
    N = Bq.shape[0]
    C = torch.empty(M, N, dtype=out, device="cuda")
    f.fp8q_mx_gemm(dev(Aq), dev(tile_scales(ea, M, K)), dev(Bq), dev(tile_scales(eb, N, K)), C)
    status_ok()
    return gemm_out_to_f64(C)


def test_gemm_scale_placement(f):
    """Unit codes, one nonzero 32-group of K at a time, distinct scale bytes
    per row and group: every output is an exact power of two that names the
    A and B scale bytes the tensor core applied."""
    M, N, K = 128, 256, 128
    rng = np.random.default_rng(1)
    ea = rng.integers(100, 140, (M, K // 32)).astype(np.uint8)
    eb = rng.integers(100, 140, (N, K // 32)).astype(np.uint8)
    for g in range(K // 32):
        Aq = np.zeros((M, K), np.uint8)
        Bq = np.zeros((N, K), np.uint8)
        Aq[:, 32 * g:32 * g + 32] = 0x38  # 1.0
        Bq[:, 32 * g:32 * g + 32] = 0x38
        C = run_gemm(f, Aq, ea, Bq, eb, torch.float32)
        want = 32.0 * np.ldexp(1.0, ea[:, g].astype(np.int64)[:, None] + eb[:, g].astype(np.int64)[None, :] - 254)
        assert np.array_equal(C, want), "group %d: first mismatch at %s" % (g, np.argwhere(C != want)[:1])


@pytest.mark.parametrize("M,N,K,out", [(128, 256, 128, torch.float32), (256, 512, 512, torch.bfloat16),
                                       (200, 384, 384, torch.float32), (77, 128, 256, torch.bfloat16),
                                       (640, 1280, 1024, torch.float32)])
def test_gemm_random_codes(f, M, N, K, out):
    rng = np.random.default_rng(M * 7 + N + K)
    Aq, Bq = rand_codes(rng, (M, K)), rand_codes(rng, (N, K))
    ea = rng.integers(117, 138, (M, K // 32)).astype(np.uint8)
    eb = rng.integers(117, 138, (N, K // 32)).astype(np.uint8)
    C = run_gemm(f, Aq, ea, Bq, eb, out)
    mi, ni = np.repeat(np.arange(M), N), np.tile(np.arange(N), M)
    ex, ab = oracle.mx_gemm_points(Aq, ea, Bq, eb, mi, ni)
    check_gemm(C.reshape(-1), ex, ab, out == torch.bfloat16, "mx %dx%dx%d" % (M, N, K))


def test_gemm_many_waves_ragged(f):
    """More tiles than CTAs (the persistent loop's accumulator handoff between
    tiles), a row tail and a half N-tile; checked on one full row per M-tile
    and one full column per N-tile."""
    M, N, K = 2100 * 2, 4608 + 128, 1152
    rng = np.random.default_rng(77)
    Aq, Bq = rand_codes(rng, (M, K)), rand_codes(rng, (N, K))
    ea = rng.integers(117, 138, (M, K // 32)).astype(np.uint8)
    eb = rng.integers(117, 138, (N, K // 32)).astype(np.uint8)
    C = run_gemm(f, Aq, ea, Bq, eb, torch.float32)
    mi, ni = sample_points(M, N)
    ex, ab = oracle.mx_gemm_points(Aq, ea, Bq, eb, mi, ni)
    check_gemm(C[mi, ni], ex, ab, False, "mx many waves")


def test_quantize_fp32_ragged_rows(f):
    x = (synth.matrix(41, 1, 333, 1280, 1.0, entry_frac=0.02, entry_scale=50.0, dtype=torch.float32) * 1e-3).cuda()
    q, s = run_quant(f, x)
    oq, oe = oracle.mx_quantize_rows(to_np(x))
    assert np.array_equal(q, oq)
    assert np.array_equal(s, tile_scales(oe, 333, 1280))


def test_gemm_zero_rows_is_noop(f):
    A = torch.empty(0, 256, dtype=torch.uint8, device="cuda")
    B = torch.zeros(128, 256, dtype=torch.uint8, device="cuda")
    sa = torch.empty(0, dtype=torch.uint8, device="cuda")
    sb = torch.zeros(f.fp8q_mx_scale_bytes(128, 256), dtype=torch.uint8, device="cuda")
    C = torch.empty(0, 128, dtype=torch.bfloat16, device="cuda")
    f.fp8q_mx_gemm(A, sa, B, sb, C)
    status_ok()


def untile(st, idx, K):
    """Scale bytes of rows `idx` read back from a tiled array
    st[K/128][row tiles][512] -> [len(idx)][K/32]."""
    r = np.asarray(idx)[:, None]
    g = np.arange(K // 32)[None, :]
    rr = r % 128
    return st[g // 4, r // 128, (rr % 32) * 16 + (rr // 32) * 4 + g % 4]


def test_quantize_then_gemm_full_size_4096x18432x7168(f):
    """The Fprop shape end to end in the MX variant: quantize X and W on the
    GPU, GEMM, then check (a) the codes and scales of every sampled row of X
    and W bit-exact against the oracle, (b) one full output row per M-tile
    and one full column per N-tile against the oracle GEMM of the GPU's
    (checked) operands."""
    X, W = synth.fprop_inputs(device="cuda")
    M, K = X.shape
    N = W.shape[0]
    qx, sx = f.mx_quantize(X)
    qw, sw = f.mx_quantize(W)
    C = f.mx_gemm(qx, sx, qw, sw, torch.bfloat16)
    status_ok()
    qx, qw = to_np(qx), to_np(qw)
    ea = untile(to_np(sx).reshape(K // 128, M // 128, 512), np.arange(M), K)
    eb = untile(to_np(sw).reshape(K // 128, N // 128, 512), np.arange(N), K)
    mi, ni = sample_points(M, N)
    rows, cols = np.unique(mi), np.unique(ni)
    oqx, oex = oracle.mx_quantize_rows(synth.bf16_bits(X[torch.from_numpy(rows).cuda()]))
    oqw, oew = oracle.mx_quantize_rows(synth.bf16_bits(W[torch.from_numpy(cols).cuda()]))
    assert np.array_equal(qx[rows], oqx) and np.array_equal(ea[rows], oex)
    assert np.array_equal(qw[cols], oqw) and np.array_equal(eb[cols], oew)
    ex, ab = oracle.mx_gemm_points(qx, ea, qw, eb, mi, ni)
    check_gemm(gemm_out_to_f64(C)[mi, ni], ex, ab, True, "mx fprop full size")
