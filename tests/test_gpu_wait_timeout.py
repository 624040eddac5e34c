"""Failure detection without a GPU fault: a kernel's bounded wait on a
barrier that nothing completes gives up, the kernel records the timeout in
the library's device error word and exits normally; the host reads
Q4K_ERR_DEVICE_TIMEOUT once, and the context keeps working."""
import numpy as np
import pytest
import torch

from oracle import q4k as O
import synth
from _gpu import pack_dev
import q4_weight_matmul_gb300 as q4k

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    q4k.build()
    assert q4k.q4k_device_error() == 0          # nothing pending before
    q4k.q4k_selftest_wait_timeout()
    assert q4k.q4k_device_error() == 5          # Q4K_ERR_DEVICE_TIMEOUT
    assert q4k.q4k_device_error() == 0          # read once, then cleared
    # the same context still computes correctly
    f = synth.q4k_fields(64, 512, 77)
    x = synth.activations(1, 512, 78)
    y = q4k.q4k_gemv(pack_dev(f), 64, 512, torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    y_ref, norm = O.gemv(f, x)
    ok, worst = O.within_tolerance(y.cpu().numpy(), y_ref, norm, 1e-4)
    assert ok, worst
    assert q4k.q4k_device_error() == 0
