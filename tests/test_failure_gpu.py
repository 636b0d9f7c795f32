"""The failure path of the bounded in-kernel waits, exercised without a GPU
fault: a wait on an mbarrier that nothing completes runs out, the kernel
records a timeout in the device error word and ends, la_check_device
reports LA_ERR_TIMEOUT (and clears it), and the context keeps computing
correct results."""
import time

import pytest
import torch

import workloads as wl
from _helpers import TOL, gpu_prefill_delta, oracle_prefill_delta, rel_err

pytestmark = pytest.mark.gpu


def test_expired_wait_is_reported_and_context_survives(cuda_lib):
    la = cuda_lib
    assert la.la_check_device() == la.LA_OK
    t0 = time.perf_counter()
    la.la_selftest_wait_timeout()
    assert la.la_check_device() == la.LA_ERR_TIMEOUT
    assert time.perf_counter() - t0 < 10.0  # the wait gives up after about a second
    # reported once, then cleared
    assert la.la_check_device() == la.LA_OK
    # the context still computes
    inp = wl.prefill_inputs([130, 64], 2, 64, 64, torch.bfloat16, False, seed=97, init_state=True)
    o, fS = gpu_prefill_delta(la, inp)
    ref_o, ref_S = oracle_prefill_delta(inp)
    assert rel_err(o.numpy(), ref_o) <= TOL[torch.bfloat16]
    assert rel_err(fS.numpy(), ref_S) <= TOL[torch.bfloat16]
