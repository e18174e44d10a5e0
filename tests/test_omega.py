"""omega drawn on the device (favor_draw_omega) against the oracle's draw of
the same definition (Philox4x64-10, Box-Muller, modified Gram-Schmidt; both
in float64, rounded to fp32 once): at most one fp32 ulp apart per element.
CPU: host validation."""
import numpy as np
import pytest

import favor_random_feature_gb300 as fv


@pytest.mark.parametrize("kw,want", [
    (dict(omega=0), fv.FAVOR_ERR_INVALID_ARG),
    (dict(omega=0x10004), fv.FAVOR_ERR_INVALID_ARG),
    (dict(H=0), fv.FAVOR_ERR_INVALID_ARG),
    (dict(m=0), fv.FAVOR_ERR_INVALID_ARG),
    (dict(kind=2), fv.FAVOR_ERR_INVALID_ARG),
    (dict(d=48), fv.FAVOR_ERR_UNSUPPORTED),
])
def test_draw_omega_host_validation(kw, want):
    fv.lib()
    a = dict(omega=0x10000, H=2, m=256, d=64, kind=1)
    a.update(kw)
    assert fv.favor_draw_omega(a["omega"], a["H"], a["m"], a["d"], a["kind"], 5, None) == want


def _ulps(got, want):
    """|got - want| in units of the fp32 spacing at want."""
    w32 = want.astype(np.float32)
    spacing = np.spacing(np.abs(w32)).astype(np.float64)
    return np.abs(got.astype(np.float64) - w32.astype(np.float64)) / spacing


@pytest.mark.gpu
@pytest.mark.parametrize("kind", [0, 1], ids=["iid", "orthogonal"])
@pytest.mark.parametrize("H,m,d", [(16, 256, 64), (3, 100, 32), (2, 300, 128), (1, 7, 32)])
def test_draw_omega_matches_oracle(kind, H, m, d):
    import torch
    import oracle
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    om = torch.full((H, m, d), float("nan"), dtype=torch.float32, device="cuda")
    rc = fv.favor_draw_omega(om, H, m, d, kind, 20241202, torch.cuda.current_stream())
    assert rc == fv.FAVOR_OK, fv.strerror(rc)
    got = om.cpu().numpy()
    want = oracle.draw_omega(H, m, d, kind, 20241202)
    assert np.isfinite(got).all()
    u = _ulps(got, want)
    assert u.max() <= 1.0, u.max()


@pytest.mark.gpu
def test_forward_with_device_drawn_omega():
    """The forward pass takes the device draw like any caller-provided omega:
    the result equals the one with the oracle's draw passed in."""
    import torch
    from favor_inputs import CAUSAL8K, make_inputs
    from parity_util import row_errors, to_device
    import oracle
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    w = CAUSAL8K
    inp = make_inputs(w, L=512, B=1, H=4)
    q, k, v, _ = to_device(inp)
    om = torch.empty((4, w.m, w.d), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    assert fv.favor_draw_omega(om, 4, w.m, w.d, 1, 77, stream) == fv.FAVOR_OK
    out = torch.empty((1, 4, 512, w.dv), dtype=torch.float32, device="cuda")
    rc = fv.favor_attn_forward(q, k, v, om, out, 1, 4, 512, w.d, w.dv, w.m, 1, 0, stream)
    assert rc == fv.FAVOR_OK, fv.strerror(rc)
    ref = oracle.forward(inp.q32, inp.k32, inp.v32, oracle.draw_omega(4, w.m, w.d, 1, 77).astype(np.float32),
                         causal=True)
    e = row_errors(out.cpu().numpy().astype(np.float64), ref)
    assert e.max() <= 2e-2 and e.mean() <= 2e-3, (e.max(), e.mean())
