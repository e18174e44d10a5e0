"""favor_attn_forward_noalloc -- the entry point for callers that must not
allocate device memory on the call path (a framework that has reserved the
GPU's memory in its own pool, a serving loop that cannot take cudaMalloc's
synchronisation).  It runs the tensor-core path on a fixed 16 MiB scratch
array inside the library.  Checked against favor_attn_forward on two calls
in a row (different inputs and modes, so stale scratch from the first call
would show in the second).  This file is collected last."""
import numpy as np
import pytest

from favor_inputs import CAUSAL8K, MAP_POSITIVE, NC4096, make_inputs
from parity_util import row_errors, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from favor_random_feature_gb300 import build
    build.build()


def test_noalloc_matches_forward_on_two_calls_in_a_row():
    import favor_random_feature_gb300 as fv
    cases = [(make_inputs(CAUSAL8K, L=2048, B=1, H=4), True),
             (make_inputs(NC4096, L=1500, B=2, H=2), False)]
    for inp, causal in cases:
        ref = run_gpu(inp, causal, MAP_POSITIVE)
        got = run_gpu(inp, causal, MAP_POSITIVE, entry=fv.favor_attn_forward_noalloc)
        e = row_errors(got, ref)
        assert e.max() <= 2e-2 and e.mean() <= 2e-3, (causal, e.max(), e.mean())


def test_noalloc_rejects_scratch_beyond_its_maximum():
    import favor_random_feature_gb300 as fv
    # B*H = 256 heads of L = 65536 need far more than 16 MiB of segment states;
    # the call must refuse before touching the (fake, far apart) pointers.
    A, Bp, C, W, O = (i << 40 for i in range(1, 6))
    rc = fv.favor_attn_forward_noalloc(A, Bp, C, W, O, 16, 16, 65536, 64, 64, 256, 1,
                                       MAP_POSITIVE)
    assert rc == fv.FAVOR_ERR_UNSUPPORTED
