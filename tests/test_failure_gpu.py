"""Failure detection on the GPU without a fault: a kernel whose bounded wait
runs out (an mbarrier nothing arrives on) must report FP8Q_ERR_TIMEOUT
through the device status word and leave the context usable.  The wait is
the same bounded mbarrier wait every pipeline of the library uses."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import status_ok

pytestmark = pytest.mark.gpu


def test_expired_wait_reports_timeout_and_context_survives():
    import fine_grained_fp8_quantize_b300 as f
    status_ok()  # nothing pending from earlier tests
    f.fp8q_selftest_wait_timeout()
    assert f.fp8q_get_device_status() == 7  # FP8Q_ERR_TIMEOUT, read and cleared
    assert f.fp8q_get_device_status() == 0
    # the context still runs the real path correctly
    A, Bt = synth.tiny_gemm_inputs(device="cuda", seed=0)
    qa, sa, _, _ = f.quantize_act(A)
    qb, sb = f.quantize_weight(Bt)
    C = f.gemm(qa, sa, qb, sb, out_dtype=torch.float32)
    status_ok()
    ex, ab, _ = oracle.gemm(qa.cpu().numpy(), sa.cpu().numpy(), qb.cpu().numpy(), sb.cpu().numpy())
    assert np.all(np.abs(C.double().cpu().numpy() - ex) <= 2e-3 * ab)
