"""Failure detection without a GPU fault.  favor_wait_expiry_check makes one
of the library's bounded mbarrier waits run out: it waits for a barrier phase
that nothing completes.  The expiry must come back through the device status
word (read and cleared by favor_get_device_status) soon after the wait's
limit, and the context must stay usable: the next forward pass still matches
the oracle.  Nothing here faults, traps or hangs the GPU."""
import time

import pytest

import favor_random_feature_gb300 as fv
from favor_inputs import CAUSAL8K, MAP_POSITIVE, make_inputs
from favor_random_feature_gb300 import build as fbuild


@pytest.mark.parametrize("limit", [0, -5, (1 << 31) + 1])
def test_limit_out_of_range_is_rejected_before_any_cuda_call(limit):
    fbuild.build()
    assert fv.favor_wait_expiry_check(limit, None) == fv.FAVOR_ERR_INVALID_ARG


@pytest.mark.gpu
def test_expired_wait_is_reported_and_the_context_stays_usable():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from parity_util import oracle_ref, row_errors, run_gpu
    fbuild.build()
    stream = torch.cuda.current_stream()
    assert fv.favor_get_device_status(stream) == fv.FAVOR_OK   # nothing pending before
    t0 = time.perf_counter()
    assert fv.favor_wait_expiry_check(1 << 21, stream) == fv.FAVOR_OK   # about a millisecond
    st = fv.favor_get_device_status(stream)                     # synchronises the stream
    elapsed = time.perf_counter() - t0
    assert st == fv.FAVOR_ERR_TIMEOUT, fv.strerror(st)
    assert elapsed < 5.0, elapsed
    assert fv.favor_get_device_status(stream) == fv.FAVOR_OK   # the read cleared it
    # the context still works: a forward pass after the expiry matches the oracle
    # (run_gpu also checks that this pass left the status word clear)
    inp = make_inputs(CAUSAL8K, L=1000, B=1, H=2)
    e = row_errors(run_gpu(inp, True, MAP_POSITIVE), oracle_ref(inp, True, MAP_POSITIVE))
    assert e.max() <= 2e-2 and e.mean() <= 2e-3, (e.max(), e.mean())
