"""The Python binding: same names as the C ABI, no CPU fallback (importing
without the built library fails), and argument checks that raise before any
call reaches the library.  No GPU needed."""
import os
import re
import shutil
import subprocess
import sys

import pytest
import torch

from conftest import ROOT

import fine_grained_fp8_quantize_b300 as f


def declared():
    src = open(os.path.join(ROOT, "include", "fp8q.h")).read()
    return sorted(set(re.findall(r"^FP8Q_API\s+(?:const\s+)?\w+\s*\*?\s*(fp8q_\w+)\s*\(", src, re.M)))


def test_binding_has_every_c_entry_point_by_name():
    for name in declared():
        assert callable(getattr(f, name)), name
        assert name in f.__all__, name


def test_import_without_the_library_fails(tmp_path):
    pkg = tmp_path / "fine_grained_fp8_quantize_b300"
    pkg.mkdir()
    shutil.copy(os.path.join(ROOT, "fine_grained_fp8_quantize_b300", "__init__.py"), pkg / "__init__.py")
    res = subprocess.run([sys.executable, "-c", "import fine_grained_fp8_quantize_b300"], cwd=tmp_path,
                         capture_output=True, text=True, timeout=300)
    assert res.returncode != 0
    assert "libfp8q.so is not built" in res.stderr


def test_argument_checks_raise_before_the_library():
    x = torch.zeros(256, 256, dtype=torch.bfloat16)
    q = torch.zeros(256, 256, dtype=torch.uint8)
    s = torch.zeros(2, 256, dtype=torch.float32)
    with pytest.raises(ValueError):  # non-contiguous
        f.fp8q_quantize_act(x.t(), q, s)
    with pytest.raises(TypeError):  # unsupported input dtype
        f.fp8q_quantize_act(torch.zeros(256, 256, dtype=torch.int32), q, s)
    with pytest.raises(ValueError):  # MX scale buffer too small
        f.fp8q_mx_quantize(x, q, torch.zeros(16, dtype=torch.uint8))
    with pytest.raises(TypeError):  # the unpromoted diagnostic writes FP32
        f.fp8q_gemm_unpromoted(q, q, torch.zeros(256, 256, dtype=torch.bfloat16))
    with pytest.raises(TypeError):  # row offsets must be int32
        f.fp8q_grouped_gemm(q, s, q.view(1, 256, 256), s, torch.zeros(256, 256, dtype=torch.bfloat16),
                            torch.zeros(2, dtype=torch.int64))


def test_status_errors_carry_code_and_text():
    e = f.Fp8qError("fp8q_gemm", 2)
    assert e.status == 2 and "fp8q_gemm" in str(e) and "shape" in str(e)
