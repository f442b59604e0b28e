"""Failure detection on the GPU without a fault: every barrier wait in the
kernels is bounded, and a wait that runs out records PKA_ERR_DEVICE_TIMEOUT
in the device error word instead of hanging or trapping.

pka_selftest_bounded_wait runs the kernels' own wait code on a barrier that
nothing completes (a short poll limit), so the timeout path runs for real;
the context must stay usable and a normal run afterwards must be clean.
"""
import numpy as np
import pytest
import torch

import paged_kv_attention_plan_gb300 as pka
from inputs import workloads as W
from tests.gpu_util import assert_parity, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

TIMEOUT = 7  # PKA_ERR_DEVICE_TIMEOUT


def test_wait_that_runs_out_records_timeout():
    assert pka.pka_get_device_error() == 0
    pka.pka_selftest_bounded_wait(False, 20)
    torch.cuda.synchronize()
    assert pka.pka_get_device_error() == TIMEOUT
    assert pka.pka_get_device_error() == 0  # read and cleared


def test_completed_wait_records_nothing():
    pka.pka_selftest_bounded_wait(True, 20)
    torch.cuda.synchronize()
    assert pka.pka_get_device_error() == 0


def test_runs_are_clean_after_a_timeout():
    pka.pka_selftest_bounded_wait(False, 5)
    torch.cuda.synchronize()
    assert pka.pka_get_device_error() == TIMEOUT
    for b in (W.worked_example(),
              W.make_paged_batch(8, np.ones(4, np.int32), [1, 300, 64, 1000], page_size=16,
                                 hq=32, hk=8, d=128, is_decode=True)):
        o, lse, _ = run_gpu(b, ("fixed", 1))  # asserts a clean device error word
        assert_parity(o, lse, *run_oracle(b))
