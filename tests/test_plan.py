"""The tensor-core launch plan, host logic only (favor_plan_info computes it
without a device).  A scan or output CTA holds most of an SM's shared memory
and TMEM, so a plan with more CTAs than SMs runs a second wave as long as the
first: the planner must keep every causal scan within one wave unless a head
cannot be cut further (one segment), and the persistent output kernel at one
CTA per SM.  The benchmark shapes' plans are pinned as well."""
import itertools

import pytest

import favor_random_feature_gb300 as fv
from favor_random_feature_gb300 import build as fbuild

GB300_SMS = 152


@pytest.fixture(scope="module", autouse=True)
def lib():
    fbuild.build()
    return fv.lib()


# (name, shape B, H, L, d, dv, m, causal, map) -> plan
#   [segments or key pieces, pieces per segment, piece states, slice CTAs,
#    value tiles, scan or output CTAs, state CTAs]
PLANS = [
    ("causal8k", (4, 16, 8192, 64, 64, 256, 1, 0), [2, 2, 2, 1, 1, 128, 128]),
    ("nc4096", (8, 12, 4096, 64, 64, 256, 0, 0), [3, 1, 3, 1, 1, 152, 288]),
    ("long64k", (1, 8, 65536, 64, 64, 256, 1, 0), [19, 1, 18, 1, 1, 152, 144]),
    ("long64k_nc", (1, 8, 65536, 64, 64, 256, 0, 0), [19, 1, 19, 1, 1, 152, 152]),
    # config 5 (d = dv = 128): whole heads at r = 128 take 4 segments (128 CTAs;
    # 5 would put 8 CTAs in a second wave), split heads 2 or 4 slices
    ("sweep16k m=128", (2, 8, 16384, 128, 128, 128, 1, 0), [4, 2, 6, 1, 2, 128, 96]),
    ("sweep16k m=64 (widened)", (2, 8, 16384, 128, 128, 64, 1, 0), [4, 2, 6, 1, 2, 128, 96]),
    ("sweep16k elu1", (2, 8, 16384, 128, 128, 128, 1, 2), [4, 2, 6, 1, 2, 128, 96]),
    ("sweep16k m=256", (2, 8, 16384, 128, 128, 256, 1, 0), [2, 4, 4, 2, 2, 128, 128]),
    ("sweep16k m=512", (2, 8, 16384, 128, 128, 512, 1, 0), [1, 1, 0, 4, 2, 128, 0]),
]


@pytest.mark.parametrize("name,shape,want", PLANS, ids=[p[0] for p in PLANS])
def test_benchmark_shapes(name, shape, want):
    rc, plan = fv.favor_plan_info(*shape, GB300_SMS)
    assert rc == fv.FAVOR_OK, fv.strerror(rc)
    assert plan == want, (name, plan)


def _shapes():
    for (B, H), L, (d, dv), (m, fmap) in itertools.product(
            [(1, 1), (1, 2), (1, 8), (2, 8), (4, 16), (8, 12), (3, 5), (16, 16), (64, 8)],
            [128, 1000, 4096, 16384, 65536],
            [(64, 64), (128, 128), (64, 128)],
            [(64, 0), (128, 0), (256, 0), (512, 0), (1024, 0), (64, 1), (128, 1), (256, 1), (128, 2), (64, 2)]):
        if fmap == 2 and m != d:
            continue
        yield B, H, L, d, dv, m, fmap


@pytest.mark.parametrize("sms", [GB300_SMS, 148, 132])
def test_one_wave(sms):
    """Causal: the scan's CTAs fit the SMs unless a head is a single segment
    (it cannot be cut further); its segments and pieces stay within the
    combine's limits.  Non-causal: the output kernel is one CTA per SM at
    most.  Over every supported shape of a grid of heads, lengths, head
    sizes and feature counts."""
    checked = 0
    for B, H, L, d, dv, m, fmap in _shapes():
        for causal in (1, 0):
            rc, plan = fv.favor_plan_info(B, H, L, d, dv, m, causal, fmap, sms)
            if rc == fv.FAVOR_ERR_UNSUPPORTED:
                continue
            assert rc == fv.FAVOR_OK
            G, pps, nstate, rs, nvb, ctas, state_ctas = plan
            shape = (B, H, L, d, dv, m, causal, fmap)
            chunks = -(-L // 128)
            assert nvb == dv // 64 and rs >= 1, shape
            if causal:
                assert 1 <= G <= min(64, chunks), (shape, plan)
                assert ctas == rs * G * nvb * B * H, (shape, plan)
                assert ctas <= sms or G == 1, (shape, plan)
                assert nstate == (G - 1) * pps, (shape, plan)
                # one segment fewer would not have filled the SMs any better
                assert G == min(64, chunks) or rs * (G + 1) * nvb * B * H > sms or \
                    -(-chunks // (G + 1)) == -(-chunks // G), (shape, plan)
            else:
                assert ctas <= sms and nstate == G >= 1, (shape, plan)
            checked += 1
    assert checked > 1000


@pytest.mark.parametrize("shape", [
    (1, 2, 64, 64, 64, 64, 1, 3),      # ReLU: SIMT kernels
    (1, 2, 64, 64, 64, 64, 0, 4),      # softmax-scaled sin/cos: SIMT kernels
    (1, 2, 64, 32, 32, 256, 1, 0),     # d = 32
    (1, 2, 64, 64, 64, 48, 1, 0),      # r = 48
    (1, 2, 64, 64, 64, 512, 0, 0),     # non-causal r = 512
])
def test_shapes_off_the_tensor_cores(shape):
    rc, _ = fv.favor_plan_info(*shape, GB300_SMS)
    assert rc == fv.FAVOR_ERR_UNSUPPORTED


def test_invalid_arguments():
    assert fv.favor_plan_info(0, 1, 64, 64, 64, 256, 1, 0, GB300_SMS)[0] == fv.FAVOR_ERR_INVALID_ARG
    assert fv.favor_plan_info(1, 1, 64, 64, 64, 256, 1, 0, 0)[0] == fv.FAVOR_ERR_INVALID_ARG
    assert fv.lib().favor_plan_info(1, 1, 64, 64, 64, 256, 1, 0, GB300_SMS, None) == fv.FAVOR_ERR_INVALID_ARG
