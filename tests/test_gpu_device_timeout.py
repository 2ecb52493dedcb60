"""The bounded waits, made to run out on purpose.

Every mbarrier wait in the kernels gives up after a fixed number of polls,
records GDR_ERR_DEVICE_TIMEOUT in the device error word and lets the kernel
leave through its normal exit.  gdr_selftest_bounded_wait runs that path on a
barrier nothing arrives on (no TMA copy or tensor-core work in flight), so the
checks here cover the whole failure-detection chain: the wait gives up, the word
is set, gdr_get_device_status reports it once and clears it, and the context
stays usable for the next call.
"""
import numpy as np
import pytest
import torch

from chunked_gated_delta_prepare_gb300 import gdr
from chunked_gated_delta_prepare_gb300.inputs import make_inputs
from gpu_helpers import all_pairs, check_forward, gpu_forward

pytestmark = pytest.mark.gpu

TIMEOUT = 7  # GDR_ERR_DEVICE_TIMEOUT


def test_wait_that_nothing_completes_reports_timeout_then_clears():
    assert gdr.gdr_get_device_status() == 0
    gdr.gdr_selftest_bounded_wait(1024, arrive=False)
    assert gdr.gdr_get_device_status() == TIMEOUT
    assert gdr.gdr_get_device_status() == 0          # read once, then cleared


def test_wait_that_completes_reports_nothing():
    assert gdr.gdr_get_device_status() == 0
    gdr.gdr_selftest_bounded_wait(1024, arrive=True)
    assert gdr.gdr_get_device_status() == 0


def test_context_stays_usable_after_a_timeout():
    gdr.gdr_selftest_bounded_wait(256, arrive=False)
    assert gdr.gdr_get_device_status() == TIMEOUT
    x = make_inputs(1, 128, 2, 128, 128, io_dtype=torch.bfloat16, with_h0=True, seed=3)
    o, hf, _ = gpu_forward(x, 64, "auto")            # asserts the status word is clear afterwards
    check_forward(x, o, hf, all_pairs(1, 2), 64, 1.0 / np.sqrt(128), "bf16")


def test_poll_limit_is_validated():
    with pytest.raises(gdr.GdrError):
        gdr.gdr_selftest_bounded_wait(0, arrive=False)
    with pytest.raises(gdr.GdrError):
        gdr.gdr_selftest_bounded_wait((1 << 22) + 1, arrive=False)
