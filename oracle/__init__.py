"""CPU oracle for fine-grained FP8 quantization and the block-scaled FP8 GEMM.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline / reference legs of ``bench.py``; never by the product
package.  It shares no code with the CUDA path.  The arithmetic lives in
``fp8q_oracle.c`` (each function there cites the passage it follows); this
module only marshals numpy arrays into it.

Functions take and return numpy arrays on the host:
  * BF16 inputs are passed as ``uint16`` arrays holding the BF16 bits, FP32 as
    ``float32``;
  * E4M3 codes are ``uint8``; scales are ``float32``;
  * scale layouts are K-block-major: ``s_row[K/128][M]``, ``s_col[M/128][K]``,
    weight ``s[N/128][K/128]``, Wgrad per-column ``sB[K/128][N]``;
  * the MX variant's scales are E8M0 bytes (``uint8``), row-major
    ``e8[rows][K/32]``.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def lib():
    """Load (building first if needed) the oracle's shared library."""
    global _lib
    if _lib is None:
        # FP8Q_ORACLE_LIB lets the mutation tests load a deliberately broken
        # copy of the oracle and check that the pins catch it
        path = os.environ.get("FP8Q_ORACLE_LIB") or _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I32 = ctypes.c_int
        L.oracle_e4m3_decode.restype = ctypes.c_float
        L.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.oracle_e4m3_encode.restype = ctypes.c_uint8
        L.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        L.oracle_e4m3_encode_array.argtypes = [P, I64, P]
        L.oracle_e4m3_decode_array.argtypes = [P, I64, P]
        L.oracle_group_scale.argtypes = [ctypes.c_float, P, P]
        L.oracle_quantize_act_rows.argtypes = [P, I32, I64, I64, P, P]
        L.oracle_quantize_act_rows_gather.argtypes = [P, I32, I64, P, I64, P, P]
        L.oracle_quantize_act_cols.argtypes = [P, I32, I64, I64, P, P]
        L.oracle_quantize_weight.argtypes = [P, I32, I64, I64, P, P]
        L.oracle_gemm_points.argtypes = [P, P, P, P, I64, I64, I64, I32, P, P, I64, P, P, P]
        L.oracle_gemm.argtypes = [P, P, P, P, I64, I64, I64, I32, P, P, P]
        L.oracle_grouped_gemm_points.argtypes = [P, P, P, P, P, I64, I64, I64, I64,
                                                 P, P, I64, P, P, P]
        L.oracle_num_threads.restype = ctypes.c_int
        L.oracle_set_num_threads.argtypes = [ctypes.c_int]
        L.oracle_mx_shared_exp.restype = ctypes.c_int
        L.oracle_mx_shared_exp.argtypes = [ctypes.c_float]
        L.oracle_mx_quantize_rows.argtypes = [P, I32, I64, I64, P, P]
        L.oracle_mx_gemm_points.argtypes = [P, P, P, P, I64, P, P, I64, P, P]
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _xin(x):
    """(array, dtype code): BF16 bits as uint16 -> 0, float32 -> 1."""
    x = np.ascontiguousarray(x)
    if x.dtype == np.uint16:
        return x, 0
    if x.dtype == np.float32:
        return x, 1
    raise TypeError("oracle input must be uint16 (BF16 bits) or float32, got %s" % x.dtype)


def num_threads():
    return lib().oracle_num_threads()


def set_num_threads(n):
    """Run later oracle calls on ``n`` OpenMP threads (timing only)."""
    lib().oracle_set_num_threads(int(n))


def e4m3_decode(codes):
    c = _c(codes, np.uint8)
    out = np.empty(c.shape, np.float32)
    lib().oracle_e4m3_decode_array(_ptr(c), c.size, _ptr(out))
    return out


def e4m3_encode(values):
    v = _c(values, np.float32)
    out = np.empty(v.shape, np.uint8)
    lib().oracle_e4m3_encode_array(_ptr(v), v.size, _ptr(out))
    return out


def group_scale(amax):
    s = ctypes.c_float()
    inv = ctypes.c_float()
    lib().oracle_group_scale(ctypes.c_float(amax), ctypes.byref(s), ctypes.byref(inv))
    return np.float32(s.value), np.float32(inv.value)


def quantize_act_rows(x):
    """1x128 groups: x[M,K] -> (q_row[M,K] u8, s_row[K/128,M] f32)."""
    x, dt = _xin(x)
    M, K = x.shape
    assert K % 128 == 0
    q = np.empty((M, K), np.uint8)
    s = np.empty((K // 128, M), np.float32)
    lib().oracle_quantize_act_rows(_ptr(x), dt, M, K, _ptr(q), _ptr(s))
    return q, s


def quantize_act_rows_gather(x, src_rows):
    """Output row r quantizes input row src_rows[r] (1x128 groups)."""
    x, dt = _xin(x)
    _, K = x.shape
    src = _c(src_rows, np.int64)
    R = src.size
    q = np.empty((R, K), np.uint8)
    s = np.empty((K // 128, R), np.float32)
    lib().oracle_quantize_act_rows_gather(_ptr(x), dt, K, _ptr(src), R, _ptr(q), _ptr(s))
    return q, s


def quantize_act_cols(x):
    """128x1 groups, transposed: x[M,K] -> (q_colT[K,M] u8, s_col[M/128,K] f32)."""
    x, dt = _xin(x)
    M, K = x.shape
    assert M % 128 == 0 and K % 128 == 0
    q = np.empty((K, M), np.uint8)
    s = np.empty((M // 128, K), np.float32)
    lib().oracle_quantize_act_cols(_ptr(x), dt, M, K, _ptr(q), _ptr(s))
    return q, s


def quantize_weight(w):
    """128x128 blocks: w[N,K] -> (q[N,K] u8, s[N/128,K/128] f32)."""
    w, dt = _xin(w)
    N, K = w.shape
    assert N % 128 == 0 and K % 128 == 0
    q = np.empty((N, K), np.uint8)
    s = np.empty((N // 128, K // 128), np.float32)
    lib().oracle_quantize_weight(_ptr(w), dt, N, K, _ptr(q), _ptr(s))
    return q, s


def gemm(Aq, sA, Bq, sB, sb_gran=128):
    """Full dense GEMM -> (C_exact f64, absref f64, C_pages f32), each [M,N]."""
    Aq = _c(Aq, np.uint8); Bq = _c(Bq, np.uint8)
    sA = _c(sA, np.float32); sB = _c(sB, np.float32)
    M, K = Aq.shape
    N = Bq.shape[0]
    ex = np.empty((M, N), np.float64)
    ab = np.empty((M, N), np.float64)
    pg = np.empty((M, N), np.float32)
    lib().oracle_gemm(_ptr(Aq), _ptr(sA), _ptr(Bq), _ptr(sB), M, N, K, sb_gran,
                      _ptr(ex), _ptr(ab), _ptr(pg))
    return ex, ab, pg


def gemm_points(Aq, sA, Bq, sB, m_idx, n_idx, sb_gran=128):
    """Dense GEMM at points -> (C_exact, absref, C_pages), each [npts]."""
    Aq = _c(Aq, np.uint8); Bq = _c(Bq, np.uint8)
    sA = _c(sA, np.float32); sB = _c(sB, np.float32)
    mi = _c(m_idx, np.int64); ni = _c(n_idx, np.int64)
    M, K = Aq.shape
    N = Bq.shape[0]
    n = mi.size
    ex = np.empty(n, np.float64)
    ab = np.empty(n, np.float64)
    pg = np.empty(n, np.float32)
    lib().oracle_gemm_points(_ptr(Aq), _ptr(sA), _ptr(Bq), _ptr(sB), M, N, K, sb_gran,
                             _ptr(mi), _ptr(ni), n, _ptr(ex), _ptr(ab), _ptr(pg))
    return ex, ab, pg


def grouped_gemm_points(Aq, sA, Bq, sB, row_offsets, m_idx, n_idx):
    """MoE grouped GEMM at points.  Bq[E,N,K], sB[E,N/128,K/128]."""
    Aq = _c(Aq, np.uint8); Bq = _c(Bq, np.uint8)
    sA = _c(sA, np.float32); sB = _c(sB, np.float32)
    off = _c(row_offsets, np.int64)
    mi = _c(m_idx, np.int64); ni = _c(n_idx, np.int64)
    T, K = Aq.shape
    E, N, _ = Bq.shape
    n = mi.size
    ex = np.empty(n, np.float64)
    ab = np.empty(n, np.float64)
    pg = np.empty(n, np.float32)
    lib().oracle_grouped_gemm_points(_ptr(Aq), _ptr(sA), _ptr(Bq), _ptr(sB), _ptr(off), E, T,
                                     N, K, _ptr(mi), _ptr(ni), n, _ptr(ex), _ptr(ab), _ptr(pg))
    return ex, ab, pg


def mx_shared_exp(amax):
    """Shared exponent of an MX group whose largest magnitude is ``amax``."""
    return lib().oracle_mx_shared_exp(ctypes.c_float(amax))


def mx_quantize_rows(x):
    """MX 1x32 groups: x[M,K] -> (q[M,K] u8 E4M3 codes, e8[M,K/32] u8 E8M0 bytes)."""
    x, dt = _xin(x)
    M, K = x.shape
    assert K % 32 == 0
    q = np.empty((M, K), np.uint8)
    e8 = np.empty((M, K // 32), np.uint8)
    lib().oracle_mx_quantize_rows(_ptr(x), dt, M, K, _ptr(q), _ptr(e8))
    return q, e8


def mx_gemm_points(Aq, ea, Bq, eb, m_idx, n_idx):
    """MX GEMM at points -> (C_exact f64, absref f64), each [npts]."""
    Aq = _c(Aq, np.uint8); Bq = _c(Bq, np.uint8)
    ea = _c(ea, np.uint8); eb = _c(eb, np.uint8)
    mi = _c(m_idx, np.int64); ni = _c(n_idx, np.int64)
    K = Aq.shape[1]
    assert Bq.shape[1] == K and ea.shape == (Aq.shape[0], K // 32) and eb.shape == (Bq.shape[0], K // 32)
    n = mi.size
    ex = np.empty(n, np.float64)
    ab = np.empty(n, np.float64)
    lib().oracle_mx_gemm_points(_ptr(Aq), _ptr(ea), _ptr(Bq), _ptr(eb), K, _ptr(mi), _ptr(ni), n,
                                _ptr(ex), _ptr(ab))
    return ex, ab
