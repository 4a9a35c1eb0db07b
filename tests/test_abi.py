"""The C-ABI library loads and exports every entry point include/fp8q.h
declares, and its host-side argument validation (which runs before any
device work) reports the documented status codes.  No GPU needed."""
import ctypes
import os
import re
import subprocess

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "fp8q.h")


def declared():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"^FP8Q_API\s+(?:const\s+)?\w+\s*\*?\s*(fp8q_\w+)\s*\(", src, re.M)))


@pytest.fixture(scope="module")
def lib():
    import fine_grained_fp8_quantize_b300 as f
    return f._lib


def test_header_declares_the_boundary():
    names = declared()
    for must in ("fp8q_quantize_act", "fp8q_quantize_weight", "fp8q_gemm", "fp8q_grouped_gemm",
                 "fp8q_gemm_ex", "fp8q_get_device_status", "fp8q_status_string"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    import fine_grained_fp8_quantize_b300 as f
    out = subprocess.run(["nm", "-D", "--defined-only", f.lib_path], capture_output=True, text=True).stdout
    exported = sorted(l.split()[-1] for l in out.splitlines() if l.split()[-1].startswith("fp8q_"))
    assert exported == declared()
    for name in declared():
        assert hasattr(lib, name)


def test_status_strings_and_version(lib):
    assert lib.fp8q_version() == 100
    for code in range(9):
        assert lib.fp8q_status_string(code)
    assert lib.fp8q_status_string(8) == b"workspace smaller than fp8q_gemm_workspace_size()"
    assert lib.fp8q_status_string(3) == b"pointer not 16-byte aligned"


# Pointers below are never dereferenced: validation rejects each call before
# it touches the device.
A = 0x10000
MIS = 0x10008
NULL = None


def test_gemm_validation(lib):
    g = lib.fp8q_gemm
    assert g(NULL, A, A, A, A, 128, 128, 128, 0, None) == 1          # null
    assert g(A, A, A, A, A, 128, 100, 128, 0, None) == 2             # N % 128
    assert g(A, A, A, A, A, 128, 128, 100, 0, None) == 2             # K % 128
    assert g(A, A, A, A, A, -1, 128, 128, 0, None) == 2              # M < 0
    assert g(A, A, A, A, A, 128, 128, 128, 7, None) == 4             # dtype
    assert g(A, A, MIS, A, A, 128, 128, 128, 0, None) == 3           # alignment
    gx = lib.fp8q_gemm_ex
    assert gx(A, A, A, A, A, 128, 128, 128, 1, 64, None) == 4        # granularity
    gw = lib.fp8q_gemm_ws
    assert gw(A, A, A, A, A, 128, 100, 128, 0, 128, A, 1 << 30, None) == 2  # N % 128
    assert gw(A, A, A, A, A, 128, 128, 128, 0, 128, MIS, 1 << 30, None) == 3  # workspace alignment
    gg = lib.fp8q_grouped_gemm
    assert gg(A, A, A, A, A, NULL, 4, 128, 128, 128, 0, None) == 1   # no offsets
    assert gg(A, A, A, A, A, A, 0, 128, 128, 128, 0, None) == 2      # E < 1
    assert gg(A, A, A, A, A, A, 5000, 128, 128, 128, 0, None) == 2   # E too large


def test_quantize_validation(lib):
    q = lib.fp8q_quantize_act
    assert q(NULL, 0, 128, 128, A, A, NULL, NULL, None) == 1
    assert q(A, 0, 128, 128, NULL, NULL, NULL, NULL, None) == 1      # no outputs
    assert q(A, 0, 128, 128, A, NULL, NULL, NULL, None) == 1         # half a pair
    assert q(A, 0, 128, 100, A, A, NULL, NULL, None) == 2            # K % 128
    assert q(A, 0, 100, 128, NULL, NULL, A, A, None) == 2            # col copy needs M % 128
    assert q(A, 2, 128, 128, A, A, NULL, NULL, None) == 4            # dtype
    assert q(MIS, 0, 128, 128, A, A, NULL, NULL, None) == 3
    w = lib.fp8q_quantize_weight
    assert w(A, 0, 100, 128, A, A, None) == 2
    assert w(A, 0, 128, 128, NULL, A, None) == 1
    wx = lib.fp8q_quantize_weight_ex
    assert wx(A, 0, 128, 128, NULL, NULL, NULL, NULL, None) == 1
    assert wx(A, 0, 128, 128, NULL, NULL, A, MIS, None) == 3
    qg = lib.fp8q_quantize_act_gather
    assert qg(A, 0, 64, 128, NULL, 10, A, A, None) == 1
    assert qg(A, 0, 0, 128, A, 10, A, A, None) == 2                  # rows from an empty x


def test_mx_validation(lib):
    sb = lib.fp8q_mx_scale_bytes
    assert sb(4096, 7168) == 56 * 32 * 512
    assert sb(1, 128) == 512 and sb(129, 256) == 2 * 2 * 512 and sb(0, 128) == 0
    assert sb(-1, 128) == 0 and sb(128, 100) == 0 and sb(128, 0) == 0
    q = lib.fp8q_mx_quantize
    assert q(NULL, 0, 128, 128, A, A, None) == 1
    assert q(A, 0, 128, 128, NULL, A, None) == 1
    assert q(A, 0, 128, 96, A, A, None) == 2                         # K % 128
    assert q(A, 0, -1, 128, A, A, None) == 2
    assert q(A, 3, 128, 128, A, A, None) == 4                        # dtype
    assert q(A, 0, 128, 128, A, MIS, None) == 3
    assert q(NULL, 0, 0, 128, NULL, NULL, None) == 0                 # empty
    g = lib.fp8q_mx_gemm
    assert g(NULL, A, A, A, A, 128, 128, 128, 0, None) == 1
    assert g(A, A, A, A, A, 128, 100, 128, 0, None) == 2             # N % 128
    assert g(A, A, A, A, A, 128, 128, 64, 0, None) == 2              # K % 128
    assert g(A, A, A, A, A, 128, 128, 128, 5, None) == 4             # dtype
    assert g(A, MIS, A, A, A, 128, 128, 128, 0, None) == 3
    assert g(NULL, NULL, NULL, NULL, NULL, 0, 128, 128, 0, None) == 0  # empty
