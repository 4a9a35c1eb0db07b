"""fine_grained_fp8_quantize_b300 -- fine-grained FP8 (E4M3) quantization and
block-scaled FP8 GEMM on B300 (sm_103a).

A thin ctypes binding over ``libfp8q.so`` (C ABI: ``include/fp8q.h``).  The
``fp8q_*`` functions here have the C names and only marshal arguments:
torch tensors supply device pointers, shapes and the current CUDA stream;
every step of the computation runs in the library's CUDA kernels.  There is
no CPU fallback: importing this package fails if the library is not built,
and every call raises ``Fp8qError`` on a non-zero status.

Layouts (see the header for the full contract):
  activations  x[M, K] -> q_row[M, K] u8, s_row[K/128, M] f32 (1x128 groups)
                       -> q_colT[K, M] u8, s_col[M/128, K] f32 (128x1, transposed)
  weights      w[N, K] -> q[N, K] u8, s[N/128, K/128] f32 (128x128 blocks)
  GEMM         C[M, N] = sum_kb sA[kb, m] * sB(kb, n) * (Aq . Bq^T)_kb
"""
import ctypes
import os

import torch

__all__ = [
    "Fp8qError", "lib_path", "FP8Q_BF16", "FP8Q_FP32",
    "fp8q_quantize_act", "fp8q_quantize_act_gather", "fp8q_quantize_weight",
    "fp8q_quantize_weight_ex", "fp8q_gemm", "fp8q_gemm_ex", "fp8q_gemm_ws", "fp8q_gemm_workspace_size",
    "fp8q_gemm_ws_static", "fp8q_gemm_unpromoted",
    "fp8q_grouped_gemm", "gemm_workspace",
    "fp8q_mx_scale_bytes", "fp8q_mx_quantize", "fp8q_mx_gemm", "fp8q_selftest_wait_timeout",
    "fp8q_get_device_status", "fp8q_status_string", "fp8q_version",
    "quantize_act", "quantize_act_gather", "quantize_weight", "gemm", "grouped_gemm", "mx_quantize", "mx_gemm",
]

FP8Q_BF16 = 0
FP8Q_FP32 = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
lib_path = os.path.join(_HERE, "libfp8q.so")


class Fp8qError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__("%s failed: status %d (%s)" % (fn, status, fp8q_status_string(status)))


def _load():
    if not os.path.exists(lib_path):
        raise ImportError("libfp8q.so is not built; run `python fine_grained_fp8_quantize_b300/build.py` "
                          "(nvcc, sm_103a)")
    L = ctypes.CDLL(lib_path)
    P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    L.fp8q_quantize_act.argtypes = [P, I32, I64, I64, P, P, P, P, P]
    L.fp8q_quantize_act_gather.argtypes = [P, I32, I64, I64, P, I64, P, P, P]
    L.fp8q_quantize_weight.argtypes = [P, I32, I64, I64, P, P, P]
    L.fp8q_quantize_weight_ex.argtypes = [P, I32, I64, I64, P, P, P, P, P]
    L.fp8q_gemm.argtypes = [P, P, P, P, P, I64, I64, I64, I32, P]
    L.fp8q_gemm_ex.argtypes = [P, P, P, P, P, I64, I64, I64, I32, I32, P]
    L.fp8q_gemm_ws.argtypes = [P, P, P, P, P, I64, I64, I64, I32, I32, P, ctypes.c_size_t, P]
    L.fp8q_gemm_ws_static.argtypes = [P, P, P, P, P, I64, I64, I64, I32, I32, P]
    L.fp8q_gemm_unpromoted.argtypes = [P, P, P, I64, I64, I64, P]
    L.fp8q_gemm_workspace_size.argtypes = []
    L.fp8q_gemm_workspace_size.restype = ctypes.c_size_t
    L.fp8q_grouped_gemm.argtypes = [P, P, P, P, P, P, ctypes.c_int32, I64, I64, I64, I32, P]
    L.fp8q_mx_scale_bytes.argtypes = [I64, I64]
    L.fp8q_mx_scale_bytes.restype = ctypes.c_size_t
    L.fp8q_mx_quantize.argtypes = [P, I32, I64, I64, P, P, P]
    L.fp8q_mx_gemm.argtypes = [P, P, P, P, P, I64, I64, I64, I32, P]
    L.fp8q_selftest_wait_timeout.argtypes = [P]
    L.fp8q_get_device_status.argtypes = [P]
    L.fp8q_status_string.restype = ctypes.c_char_p
    L.fp8q_status_string.argtypes = [I32]
    for name in ("fp8q_quantize_act", "fp8q_quantize_act_gather", "fp8q_quantize_weight",
                 "fp8q_quantize_weight_ex", "fp8q_gemm", "fp8q_gemm_ex", "fp8q_gemm_ws", "fp8q_gemm_ws_static",
                 "fp8q_gemm_unpromoted", "fp8q_grouped_gemm", "fp8q_mx_quantize", "fp8q_mx_gemm",
                 "fp8q_selftest_wait_timeout",
                 "fp8q_get_device_status", "fp8q_version"):
        getattr(L, name).restype = I32
    return L


_lib = _load()


def fp8q_status_string(status):
    return _lib.fp8q_status_string(int(status)).decode()


def fp8q_version():
    return _lib.fp8q_version()


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if isinstance(stream, torch.cuda.Stream) else int(stream)


def _in_dtype(x):
    if x.dtype == torch.bfloat16:
        return FP8Q_BF16
    if x.dtype == torch.float32:
        return FP8Q_FP32
    raise TypeError("input must be bfloat16 or float32, got %s" % x.dtype)


def _out_dtype(c):
    if c.dtype == torch.bfloat16:
        return FP8Q_BF16
    if c.dtype == torch.float32:
        return FP8Q_FP32
    raise TypeError("output must be bfloat16 or float32, got %s" % c.dtype)


def _check(fn, st):
    if st != 0:
        raise Fp8qError(fn, st)


def _contig(*ts):
    for t in ts:
        if t is not None and not t.is_contiguous():
            raise ValueError("tensors passed to libfp8q must be contiguous")


# --------------------------------------------------------------------------
# C-named entry points: marshal tensors to pointers, sizes and the stream.
# --------------------------------------------------------------------------

def fp8q_quantize_act(x, q_row=None, s_row=None, q_colT=None, s_col=None, stream=None):
    _contig(x, q_row, s_row, q_colT, s_col)
    M, K = x.shape
    _check("fp8q_quantize_act", _lib.fp8q_quantize_act(
        _ptr(x), _in_dtype(x), M, K, _ptr(q_row), _ptr(s_row), _ptr(q_colT), _ptr(s_col), _stream(stream)))


def fp8q_quantize_act_gather(x, src_rows, q_row, s_row, stream=None):
    _contig(x, src_rows, q_row, s_row)
    if src_rows.dtype != torch.int32:
        raise TypeError("src_rows must be int32")
    M, K = x.shape
    _check("fp8q_quantize_act_gather", _lib.fp8q_quantize_act_gather(
        _ptr(x), _in_dtype(x), M, K, _ptr(src_rows), src_rows.numel(), _ptr(q_row), _ptr(s_row),
        _stream(stream)))


def fp8q_quantize_weight(w, q, s, stream=None):
    _contig(w, q, s)
    N, K = w.shape
    _check("fp8q_quantize_weight", _lib.fp8q_quantize_weight(
        _ptr(w), _in_dtype(w), N, K, _ptr(q), _ptr(s), _stream(stream)))


def fp8q_quantize_weight_ex(w, q=None, s=None, q_t=None, s_t=None, stream=None):
    _contig(w, q, s, q_t, s_t)
    N, K = w.shape
    _check("fp8q_quantize_weight_ex", _lib.fp8q_quantize_weight_ex(
        _ptr(w), _in_dtype(w), N, K, _ptr(q), _ptr(s), _ptr(q_t), _ptr(s_t), _stream(stream)))


def fp8q_gemm(Aq, sA, Bq, sB, C, stream=None):
    _contig(Aq, sA, Bq, sB, C)
    M, K = Aq.shape
    N = Bq.shape[0]
    _check("fp8q_gemm", _lib.fp8q_gemm(
        _ptr(Aq), _ptr(sA), _ptr(Bq), _ptr(sB), _ptr(C), M, N, K, _out_dtype(C), _stream(stream)))


def fp8q_gemm_ex(Aq, sA, Bq, sB, C, sb_gran_n, stream=None):
    _contig(Aq, sA, Bq, sB, C)
    M, K = Aq.shape
    N = Bq.shape[0]
    _check("fp8q_gemm_ex", _lib.fp8q_gemm_ex(
        _ptr(Aq), _ptr(sA), _ptr(Bq), _ptr(sB), _ptr(C), M, N, K, _out_dtype(C), int(sb_gran_n),
        _stream(stream)))


def fp8q_gemm_workspace_size():
    return int(_lib.fp8q_gemm_workspace_size())


def fp8q_gemm_ws(Aq, sA, Bq, sB, C, sb_gran_n, workspace, stream=None):
    _contig(Aq, sA, Bq, sB, C, workspace)
    M, K = Aq.shape
    N = Bq.shape[0]
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("fp8q_gemm_ws", _lib.fp8q_gemm_ws(
        _ptr(Aq), _ptr(sA), _ptr(Bq), _ptr(sB), _ptr(C), M, N, K, _out_dtype(C), int(sb_gran_n),
        _ptr(workspace), nbytes, _stream(stream)))


def fp8q_gemm_ws_static(Aq, sA, Bq, sB, C, sb_gran_n, stream=None):
    """fp8q_gemm_ws on the library's own fixed scratch: allocates nothing."""
    _contig(Aq, sA, Bq, sB, C)
    M, K = Aq.shape
    N = Bq.shape[0]
    _check("fp8q_gemm_ws_static", _lib.fp8q_gemm_ws_static(
        _ptr(Aq), _ptr(sA), _ptr(Bq), _ptr(sB), _ptr(C), M, N, K, _out_dtype(C), int(sb_gran_n),
        _stream(stream)))


def fp8q_gemm_unpromoted(Aq, Bq, C, stream=None):
    """Diagnostic: C = Aq . Bq^T (decoded codes) accumulated over the whole K
    inside the tensor core, without promotion or scales; C is FP32."""
    _contig(Aq, Bq, C)
    if C.dtype != torch.float32:
        raise TypeError("fp8q_gemm_unpromoted writes FP32")
    M, K = Aq.shape
    N = Bq.shape[0]
    _check("fp8q_gemm_unpromoted", _lib.fp8q_gemm_unpromoted(_ptr(Aq), _ptr(Bq), _ptr(C), M, N, K, _stream(stream)))


def fp8q_grouped_gemm(Aq, sA, Bq, sB, C, row_offsets, stream=None):
    _contig(Aq, sA, Bq, sB, C, row_offsets)
    if row_offsets.dtype != torch.int32:
        raise TypeError("row_offsets must be int32")
    T, K = Aq.shape
    E, N, _ = Bq.shape
    _check("fp8q_grouped_gemm", _lib.fp8q_grouped_gemm(
        _ptr(Aq), _ptr(sA), _ptr(Bq), _ptr(sB), _ptr(C), _ptr(row_offsets), E, T, N, K,
        _out_dtype(C), _stream(stream)))


def fp8q_mx_scale_bytes(rows, K):
    return _lib.fp8q_mx_scale_bytes(rows, K)


def fp8q_mx_quantize(x, q, s, stream=None):
    """MX 1x32 quantization: x[rows,K] -> q[rows,K] codes, s tiled E8M0 scales (uint8)."""
    _contig(x, q, s)
    rows, K = x.shape
    if s is not None and s.numel() < fp8q_mx_scale_bytes(rows, K):
        raise ValueError("scale buffer smaller than fp8q_mx_scale_bytes(rows, K)")
    _check("fp8q_mx_quantize", _lib.fp8q_mx_quantize(_ptr(x), _in_dtype(x), rows, K, _ptr(q), _ptr(s),
                                                     _stream(stream)))


def fp8q_mx_gemm(Aq, sA, Bq, sB, C, stream=None):
    _contig(Aq, sA, Bq, sB, C)
    M, K = Aq.shape
    N = Bq.shape[0]
    if sA.numel() < fp8q_mx_scale_bytes(M, K) or sB.numel() < fp8q_mx_scale_bytes(N, K):
        raise ValueError("scale buffer smaller than fp8q_mx_scale_bytes")
    _check("fp8q_mx_gemm", _lib.fp8q_mx_gemm(_ptr(Aq), _ptr(sA), _ptr(Bq), _ptr(sB), _ptr(C), M, N, K,
                                             _out_dtype(C), _stream(stream)))


def fp8q_selftest_wait_timeout(stream=None):
    """Failure-detection self-test: a kernel whose bounded wait expires
    (about 2 s); afterwards fp8q_get_device_status() reports the timeout."""
    _check("fp8q_selftest_wait_timeout", _lib.fp8q_selftest_wait_timeout(_stream(stream)))


def fp8q_get_device_status(stream=None):
    return _lib.fp8q_get_device_status(_stream(stream))


# --------------------------------------------------------------------------
# Conveniences that allocate the outputs with torch (device memory only).
# --------------------------------------------------------------------------

def quantize_act(x, row=True, col=False, stream=None):
    """-> (q_row, s_row, q_colT, s_col); skipped outputs are None."""
    M, K = x.shape
    dev = x.device
    q_row = torch.empty(M, K, dtype=torch.uint8, device=dev) if row else None
    s_row = torch.empty(K // 128, M, dtype=torch.float32, device=dev) if row else None
    q_colT = torch.empty(K, M, dtype=torch.uint8, device=dev) if col else None
    s_col = torch.empty(M // 128, K, dtype=torch.float32, device=dev) if col else None
    fp8q_quantize_act(x, q_row, s_row, q_colT, s_col, stream)
    return q_row, s_row, q_colT, s_col


def quantize_act_gather(x, src_rows, stream=None):
    R = src_rows.numel()
    K = x.shape[1]
    q = torch.empty(R, K, dtype=torch.uint8, device=x.device)
    s = torch.empty(K // 128, R, dtype=torch.float32, device=x.device)
    fp8q_quantize_act_gather(x, src_rows, q, s, stream)
    return q, s


def quantize_weight(w, transposed=False, stream=None):
    """-> (q, s) or, with transposed=True, (q, s, q_t, s_t)."""
    N, K = w.shape
    dev = w.device
    q = torch.empty(N, K, dtype=torch.uint8, device=dev)
    s = torch.empty(N // 128, K // 128, dtype=torch.float32, device=dev)
    if not transposed:
        fp8q_quantize_weight(w, q, s, stream)
        return q, s
    q_t = torch.empty(K, N, dtype=torch.uint8, device=dev)
    s_t = torch.empty(K // 128, N // 128, dtype=torch.float32, device=dev)
    fp8q_quantize_weight_ex(w, q, s, q_t, s_t, stream)
    return q, s, q_t, s_t


def gemm_workspace(device=None):
    """A zero-filled stream-K workspace for fp8q_gemm_ws on `device`."""
    n = fp8q_gemm_workspace_size()
    if n == 0:
        raise Fp8qError("fp8q_gemm_workspace_size", 5)
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def gemm(Aq, sA, Bq, sB, out_dtype=torch.bfloat16, sb_gran_n=128, workspace=None, stream=None):
    M = Aq.shape[0]
    N = Bq.shape[0]
    C = torch.empty(M, N, dtype=out_dtype, device=Aq.device)
    if workspace is not None:
        fp8q_gemm_ws(Aq, sA, Bq, sB, C, sb_gran_n, workspace, stream)
    elif sb_gran_n == 128:
        fp8q_gemm(Aq, sA, Bq, sB, C, stream)
    else:
        fp8q_gemm_ex(Aq, sA, Bq, sB, C, sb_gran_n, stream)
    return C


def grouped_gemm(Aq, sA, Bq, sB, row_offsets, out_dtype=torch.bfloat16, stream=None):
    C = torch.empty(Aq.shape[0], Bq.shape[1], dtype=out_dtype, device=Aq.device)
    fp8q_grouped_gemm(Aq, sA, Bq, sB, C, row_offsets, stream)
    return C


def mx_quantize(x, stream=None):
    """MX variant: -> (q [rows, K] uint8 codes, s tiled E8M0 scales, uint8)."""
    rows, K = x.shape
    q = torch.empty(rows, K, dtype=torch.uint8, device=x.device)
    s = torch.empty(fp8q_mx_scale_bytes(rows, K), dtype=torch.uint8, device=x.device)
    fp8q_mx_quantize(x, q, s, stream)
    return q, s


def mx_gemm(Aq, sA, Bq, sB, out_dtype=torch.bfloat16, stream=None):
    C = torch.empty(Aq.shape[0], Bq.shape[0], dtype=out_dtype, device=Aq.device)
    fp8q_mx_gemm(Aq, sA, Bq, sB, C, stream)
    return C
