"""The backward pass (favor_attn_backward / _f32) against the float64
oracle's gradients (oracle.backward, pinned to finite differences of the
forward pass), row by row: for every row t of dq, dk, dv (a token) and of
domega (a projection),

    e_t = |G_t - G_ref_t| / max(|G_ref_t|, 1e-2 rms_t |G_ref_t|),

the normwise per-row error of the forward parity tests, with a floor at
1e-2 of the tensor's root-mean-square row norm: a row whose exact gradient
vanishes (dq of the first causal row: out_0 = v_0 whatever q_0) is scored
against the others' scale instead of against rounding noise (its error
must still stay below 2e-4 of the rms row).  Bars: max_t
e_t <= 2e-2 (the forward bf16 bar's) and mean_t e_t <= 2e-5.  The SIMT
kernels compute in fp32 on the inputs' values (bf16 inputs are exact in
fp32), so one bar serves both entry points.  Measured on the GB300: mean row
errors of 1e-7 to 4e-6 (3.3e-6 for dq at the full benchmark shape); single
rows of dq reach 2e-3 to 7e-3 where the feature terms of a small-gradient
row cancel (early causal rows, d = 128).  A wrong, missing or misplaced term
moves a row by 1e-1 or more, so the max bar still catches it, and the mean
bar sits five times above the worst measured mean.  CPU: host validation."""
import numpy as np
import pytest

import favor_random_feature_gb300 as fv
from favor_inputs import (CAUSAL8K, MAP_ELU1, MAP_POSITIVE, MAP_RELU, MAP_TRIG, MAP_TRIG_SOFTMAX, NC4096,
                          make_inputs)

NO_OMEGA = (MAP_ELU1, MAP_RELU)
GRAD_MAX, GRAD_MEAN = 2e-2, 2e-5
ROW_FLOOR = 1e-2


A, K, V, W, G, DQ, DK, DV, DW = (0x10000 * i for i in range(1, 10))


@pytest.mark.parametrize("kw,want", [
    (dict(dq=0), fv.FAVOR_ERR_INVALID_ARG),
    (dict(dout=0), fv.FAVOR_ERR_INVALID_ARG),
    (dict(dk=DK + 4), fv.FAVOR_ERR_INVALID_ARG),
    (dict(dv=DQ + 64), fv.FAVOR_ERR_INVALID_ARG),        # outputs overlap
    (dict(dq=K), fv.FAVOR_ERR_INVALID_ARG),              # an output over an input
    (dict(d=48), fv.FAVOR_ERR_UNSUPPORTED),
    (dict(causal=2), fv.FAVOR_ERR_INVALID_ARG),
])
def test_backward_host_validation(kw, want):
    fv.lib()
    a = dict(q=A, k=K, v=V, omega=W, dout=G, dq=DQ, dk=DK, dv=DV, domega=DW, B=1, H=1, L=16, d=64, dv_=64,
             m=64, causal=1, feature_map=MAP_POSITIVE)
    a.update(kw)
    for fn in (fv.favor_attn_backward, fv.favor_attn_backward_f32):
        rc = fn(a["q"], a["k"], a["v"], a["omega"], a["dout"], a["dq"], a["dk"], a["dv"], a["domega"], a["B"],
                a["H"], a["L"], a["d"], a["dv_"], a["m"], a["causal"], a["feature_map"], None)
        assert rc == want, (fn.__name__, kw, fv.strerror(rc))


def _run(inp, g, causal, fmap, f32):
    """favor_attn_backward(_f32) on the inputs; returns (dq, dk, dv, dw) as float64."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from favor_random_feature_gb300 import build
    build.build()
    w = inp.w
    bf16 = w.dtype == "bf16" and not f32
    if bf16:
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
        q, k, v = dev(inp.q), dev(inp.k), dev(inp.v)
    else:
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()
        q, k, v = dev(inp.q32), dev(inp.k32), dev(inp.v32)
    m = w.d if fmap in NO_OMEGA else w.m
    om = None if fmap in NO_OMEGA else torch.from_numpy(np.ascontiguousarray(inp.omega, dtype=np.float32)).cuda()
    gd = torch.from_numpy(np.ascontiguousarray(g, dtype=np.float32)).cuda()
    nan = lambda shape: torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")
    dq, dk, dv = nan((w.B, w.H, w.L, w.d)), nan((w.B, w.H, w.L, w.d)), nan((w.B, w.H, w.L, w.dv))
    dw = None if om is None else nan((w.H, m, w.d))
    fn = fv.favor_attn_backward if bf16 else fv.favor_attn_backward_f32
    stream = torch.cuda.current_stream()
    rc = fn(q, k, v, om, gd, dq, dk, dv, dw, w.B, w.H, w.L, w.d, w.dv, m, int(causal), fmap, stream)
    assert rc == fv.FAVOR_OK, fv.strerror(rc)
    st = fv.favor_get_device_status(stream)
    assert st == fv.FAVOR_OK, fv.strerror(st)
    to = lambda t: None if t is None else t.cpu().numpy().astype(np.float64)
    return to(dq), to(dk), to(dv), to(dw)


def row_errors(got, ref):
    """Per-row normwise error with a floor at ROW_FLOOR x the rms row norm."""
    a = got.reshape(-1, got.shape[-1])
    b = ref.reshape(-1, ref.shape[-1])
    nb = np.linalg.norm(b, axis=1)
    floor = ROW_FLOOR * np.sqrt(np.mean(nb ** 2))
    return np.linalg.norm(a - b, axis=1) / np.maximum(nb, floor)


def _check(got, ref, bar_max=GRAD_MAX, bar_mean=GRAD_MEAN):
    names = ("dq", "dk", "dv", "dw")
    for name, a, b in zip(names, got, ref):
        if b is None:
            assert a is None
            continue
        assert np.isfinite(a).all(), name
        e = row_errors(a, b)
        assert e.max() <= bar_max and e.mean() <= bar_mean, (name, e.max(), e.mean())


CASES = [
    (MAP_POSITIVE, 64), (MAP_TRIG, 32), (MAP_ELU1, None), (MAP_RELU, None), (MAP_TRIG_SOFTMAX, 32),
]


@pytest.mark.gpu
@pytest.mark.parametrize("f32", [False, True], ids=["bf16", "f32"])
@pytest.mark.parametrize("causal", [False, True], ids=["noncausal", "causal"])
@pytest.mark.parametrize("fmap,m", CASES, ids=["positive", "trig", "elu1", "relu", "trig_softmax"])
def test_backward_matches_oracle(fmap, m, causal, f32):
    import oracle
    w = NC4096.with_(feature_map=fmap, omega="iid", m=m or 64, dtype="bf16")
    if fmap in NO_OMEGA:
        w = w.with_(m=w.d)
    inp = make_inputs(w, L=200, B=2, H=3)
    if fmap in (MAP_TRIG, MAP_TRIG_SOFTMAX):
        # small q, k keep the sin/cos denominators away from zero
        from parity_util import scaled_inputs
        inp = scaled_inputs(inp, 0.3)
    g = np.random.default_rng(71).standard_normal((2, 3, 200, w.dv))
    got = _run(inp, g, causal, fmap, f32)
    ref = oracle.backward(inp.q32, inp.k32, inp.v32, None if fmap in NO_OMEGA else inp.omega, g, causal, fmap)
    _check(got, ref)


@pytest.mark.gpu
@pytest.mark.parametrize("causal", [False, True], ids=["noncausal", "causal"])
@pytest.mark.parametrize("fmap", [MAP_POSITIVE, MAP_ELU1], ids=["positive", "elu1"])
@pytest.mark.parametrize("d,dv,m", [(32, 32, 64), (64, 128, 64), (128, 128, 128)],
                         ids=["d32", "d64-dv128", "d128"])
def test_backward_head_dims(d, dv, m, fmap, causal):
    """The other instances of the templated backward kernels: d = dv = 32,
    dv = 128 (the 156 KB shared-memory launch shape of the chunk kernel) and
    d = dv = 128."""
    import oracle
    w = NC4096.with_(feature_map=fmap, omega="iid", m=m, dtype="bf16", d=d, dv=dv)
    if fmap in NO_OMEGA:
        w = w.with_(m=w.d)
    inp = make_inputs(w, L=200, B=2, H=3)
    g = np.random.default_rng(73).standard_normal((2, 3, 200, w.dv))
    got = _run(inp, g, causal, fmap, False)
    ref = oracle.backward(inp.q32, inp.k32, inp.v32, None if fmap in NO_OMEGA else inp.omega, g, causal, fmap)
    _check(got, ref)


@pytest.mark.gpu
def test_backward_full_size_sampled_heads():
    """The benchmark shape (B=4, H=16, L=8192, d=dv=64, m=256, causal): two
    heads (all four batches, so their omega gradients are complete) against
    the oracle, at the same per-row bars as the reduced shapes."""
    import oracle
    w = CAUSAL8K
    inp = make_inputs(w)
    g = np.random.default_rng(72).standard_normal((w.B, w.H, w.L, w.dv)).astype(np.float32)
    got = _run(inp, g, True, MAP_POSITIVE, False)
    hs = [5, 11]
    ref = oracle.backward(inp.q32[:, hs], inp.k32[:, hs], inp.v32[:, hs], inp.omega[hs], g[:, hs].astype(np.float64),
                          True, MAP_POSITIVE)
    _check((got[0][:, hs], got[1][:, hs], got[2][:, hs], got[3][hs]), ref)
