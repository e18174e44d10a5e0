"""The range of the tensor-core path (fp16 MMA operands, see favor.h,
"Range of the tensor-core path").

Inputs that stay inside it -- keys whose norms vary by a factor of five
within a head, a large-norm key placed late in a 128-token chunk after small
ones, values near +-6e4 -- must meet the bf16 parity bar against the float64
oracle with a clean device status.  Inputs that leave it must not pass
silently: the call completes and the device status word reads
FAVOR_ERR_RANGE, while the fp32 entry point computes the same values within
the fp32 bar."""
import numpy as np
import pytest

from favor_inputs import CAUSAL8K, MAP_POSITIVE, SWEEP16K, bf16_bits, bf16_to_f32, make_inputs
from parity_util import oracle_ref, row_errors, run_gpu, to_device

pytestmark = pytest.mark.gpu

BF16_MAX, BF16_MEAN, F32_MAX = 2e-2, 2e-3, 1e-4
L = 1024


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from favor_random_feature_gb300 import build
    build.build()


def _with(inp, q=None, k=None, v=None):
    """The same inputs with q, k or v replaced (re-rounded to bf16)."""
    import copy
    out = copy.copy(inp)
    for name, x in (("q", q), ("k", k), ("v", v)):
        if x is not None:
            bits = bf16_bits(x.astype(np.float32))
            setattr(out, name, bits)
            setattr(out, name + "32", bf16_to_f32(bits))
    return out


def _call_status(inp, causal):
    """favor_attn_forward on the inputs; returns (out, device status)."""
    import torch
    import favor_random_feature_gb300 as fv
    w = inp.w
    q, k, v, om = to_device(inp)
    out = torch.empty((w.B, w.H, w.L, w.dv), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    fv.favor_get_device_status(stream)   # start from a clear status word
    rc = fv.favor_attn_forward(q, k, v, om, out, w.B, w.H, w.L, w.d, w.dv, w.m, int(causal), MAP_POSITIVE,
                               stream)
    assert rc == fv.FAVOR_OK, fv.strerror(rc)
    return out.cpu().numpy().astype(np.float64), fv.favor_get_device_status(stream)


def _f32_entry(inp, causal):
    """favor_attn_forward_f32 on the exact values (bf16 widened to fp32)."""
    import copy
    f = copy.copy(inp)
    f.w = inp.w.with_(dtype="f32")
    f.q, f.k, f.v = inp.q32, inp.k32, inp.v32
    return run_gpu(f, causal, MAP_POSITIVE)


def wide_spread_inputs(w=CAUSAL8K):
    """Keys in blocks of 128 scaled x0.5, x1 and x2.5 around N(0,1) d^-1/4, one
    key per chunk scaled x4 at position 120 (after the chunk's other keys), and
    values with a few entries near +-6e4."""
    inp = make_inputs(w, L=L, B=1, H=2)
    k = inp.k32.copy()
    scale = np.resize(np.repeat([0.5, 1.0, 2.5], 128), L).astype(np.float32)
    k *= scale[None, None, :, None]
    k[:, :, 120::128] *= 4.0
    v = inp.v32.copy()
    rng = np.random.default_rng(123)
    idx = rng.choice(L, 6, replace=False)
    v[0, 0, idx, rng.integers(0, v.shape[-1], 6)] = np.float32(6.0e4) * np.sign(rng.standard_normal(6)).astype(np.float32)
    return _with(inp, k=k, v=v)


@pytest.mark.parametrize("causal,w", [(True, CAUSAL8K), (False, CAUSAL8K), (True, SWEEP16K)],
                         ids=["causal", "noncausal", "causal-split"])
def test_wide_key_norm_spread_meets_the_bar(causal, w):
    import favor_random_feature_gb300 as fv
    inp = wide_spread_inputs(w)
    out, st = _call_status(inp, causal)
    assert st == fv.FAVOR_OK, fv.strerror(st)
    e = row_errors(out, oracle_ref(inp, causal, MAP_POSITIVE))
    assert e.max() <= BF16_MAX and e.mean() <= BF16_MEAN, (e.max(), e.mean())


@pytest.mark.parametrize("causal,w", [(True, CAUSAL8K), (False, CAUSAL8K), (True, SWEEP16K)],
                         ids=["causal", "noncausal", "causal-split"])
def test_key_on_a_projection_row_reports_range(causal, w):
    """A key along the longest row w_f of omega, k = a w_f, has the feature
    exp(|w_f|^2 (a - a^2/2)) against about e^0 for the other keys: a = 1 at
    d = 64 (|w_f|^2 / 2 ~ 48), a < 1 at d = 128 so that the gap is also e^48
    (at a = 1 it would be ~e^90, past fp32's own e^-87).  The other keys'
    features underflow fp16 at its reference while queries that barely see
    it still need them.  The call must say so; the fp32 entry point computes
    the same values within the fp32 bar."""
    import favor_random_feature_gb300 as fv
    inp = make_inputs(w, L=L, B=1, H=2)
    k = inp.k32.copy()
    for h in range(2):
        f = int(np.argmax(np.linalg.norm(inp.omega[h], axis=1)))
        n2 = float(np.sum(inp.omega[h, f].astype(np.float64) ** 2))
        gap = min(n2 / 2, 48.5)
        a = 1.0 - np.sqrt(1.0 - 2.0 * gap / n2)
        k[0, h, 500] = a * inp.omega[h, f]
    inp = _with(inp, k=k)
    _, st = _call_status(inp, causal)
    assert st == fv.FAVOR_ERR_RANGE, fv.strerror(st)
    e = row_errors(_f32_entry(inp, causal), oracle_ref(inp, causal, MAP_POSITIVE))
    assert e.max() <= F32_MAX, e.max()


@pytest.mark.parametrize("which", ["q", "k", "v"])
@pytest.mark.parametrize("w", [CAUSAL8K, SWEEP16K], ids=["whole", "split"])
def test_operand_beyond_fp16_reports_range(which, w):
    """A value of 7e4 (bf16 69632) has no finite fp16 image."""
    import favor_random_feature_gb300 as fv
    inp = make_inputs(w, L=300, B=1, H=2)
    x = getattr(inp, which + "32").copy()
    x[0, 1, 77, 5] = 7.0e4
    inp = _with(inp, **{which: x})
    for causal in ((True, False) if w is CAUSAL8K else (True,)):
        _, st = _call_status(inp, causal)
        assert st == fv.FAVOR_ERR_RANGE, (which, causal, fv.strerror(st))


def test_status_is_clean_after_a_range_report():
    """The status word is cleared by reading it: the next in-range call reports OK."""
    import favor_random_feature_gb300 as fv
    inp = make_inputs(CAUSAL8K, L=300, B=1, H=2)
    v = inp.v32.copy()
    v[0, 0, 3, 3] = 7.0e4
    _, st = _call_status(_with(inp, v=v), True)
    assert st == fv.FAVOR_ERR_RANGE
    out, st = _call_status(inp, True)
    assert st == fv.FAVOR_OK, fv.strerror(st)
    e = row_errors(out, oracle_ref(inp, True, MAP_POSITIVE))
    assert e.max() <= BF16_MAX and e.mean() <= BF16_MEAN
