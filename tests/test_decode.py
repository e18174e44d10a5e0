"""The carried state and the one-token decode step (Performer study notes,
"Case 2": S_i, z_i are running sums, so a new token costs O(r d)).

GPU parity: favor_attn_state over a prefix of L0 keys, then T calls of
favor_attn_decode, against the float64 oracle: the state against
oracle.state (per head, |S - S_ref|_F / |S_ref|_F over [S | z]) and the
decode outputs against the causal rows L0 .. L0+T-1 of oracle.forward on the
whole sequence (the recurrence the oracle states), with the forward pass's
tolerances (fp32 1e-4; bf16 max 2e-2, mean 2e-3 normwise per row).
CPU: host validation of the new entry points."""
import numpy as np
import pytest

import favor_random_feature_gb300 as fv
from favor_inputs import (CAUSAL8K, DEMO64, LONG64K, MAP_ELU1, MAP_POSITIVE, MAP_RELU, MAP_TRIG,
                          MAP_TRIG_SOFTMAX, make_inputs)

NO_OMEGA = (MAP_ELU1, MAP_RELU)
from parity_util import row_errors

F32_MAX = 1e-4
BF16_MAX = 2e-2
BF16_MEAN = 2e-3
STATE_BF16 = 2e-3     # fp16 features, fp32 sums
STATE_F32 = 1e-5


# ---------------------------------------------------------------------------
# host side (no GPU)
# ---------------------------------------------------------------------------
def test_state_floats():
    assert fv.favor_state_floats(64, 64, 256, MAP_POSITIVE) == 256 * 66
    assert fv.favor_state_floats(64, 128, 256, MAP_TRIG) == 512 * 130
    assert fv.favor_state_floats(64, 32, 64, MAP_ELU1) == 64 * 34
    assert fv.favor_state_floats(64, 64, 32, MAP_ELU1) == -1
    assert fv.favor_state_floats(48, 64, 256, MAP_POSITIVE) == -1


A, K, V, W, S, O = 0x10000, 0x20000, 0x30000, 0x40000, 0x1000000, 0x50000


@pytest.mark.parametrize("kw,want", [
    (dict(state=0), fv.FAVOR_ERR_INVALID_ARG),
    (dict(state=S + 4), fv.FAVOR_ERR_INVALID_ARG),
    (dict(q=0), fv.FAVOR_ERR_INVALID_ARG),
    (dict(omega=0), fv.FAVOR_ERR_INVALID_ARG),
    (dict(out=S + 64), fv.FAVOR_ERR_INVALID_ARG),        # out inside the state
    (dict(state=K), fv.FAVOR_ERR_INVALID_ARG),           # state over an input
    (dict(m=1024, feature_map=MAP_TRIG), fv.FAVOR_ERR_UNSUPPORTED),   # r = 2048
    (dict(d=48), fv.FAVOR_ERR_UNSUPPORTED),
    (dict(m=100), fv.FAVOR_ERR_UNSUPPORTED),
    (dict(m=32, feature_map=MAP_ELU1), fv.FAVOR_ERR_INVALID_ARG),
    (dict(B=0), fv.FAVOR_ERR_INVALID_ARG),
])
def test_decode_host_validation(kw, want):
    fv.lib()
    a = dict(q=A, k=K, v=V, omega=W, state=S, out=O, B=1, H=2, d=64, dv=64, m=256,
             feature_map=MAP_POSITIVE)
    a.update(kw)
    for fn in (fv.favor_attn_decode, fv.favor_attn_decode_f32):
        rc = fn(a["q"], a["k"], a["v"], a["omega"], a["state"], a["out"], a["B"], a["H"], a["d"],
                a["dv"], a["m"], a["feature_map"], None)
        assert rc == want, (fn.__name__, kw, fv.strerror(rc))


@pytest.mark.parametrize("kw,want", [
    (dict(state=0), fv.FAVOR_ERR_INVALID_ARG),
    (dict(k=0), fv.FAVOR_ERR_INVALID_ARG),
    (dict(L=-1), fv.FAVOR_ERR_INVALID_ARG),
    (dict(state=V), fv.FAVOR_ERR_INVALID_ARG),
    (dict(dv=96), fv.FAVOR_ERR_UNSUPPORTED),
])
def test_state_host_validation(kw, want):
    fv.lib()
    a = dict(k=K, v=V, omega=W, state=S, B=1, H=2, L=64, d=64, dv=64, m=256,
             feature_map=MAP_POSITIVE)
    a.update(kw)
    for fn in (fv.favor_attn_state, fv.favor_attn_state_f32):
        rc = fn(a["k"], a["v"], a["omega"], a["state"], a["B"], a["H"], a["L"], a["d"], a["dv"],
                a["m"], a["feature_map"], None)
        assert rc == want, (fn.__name__, kw, fv.strerror(rc))


# ---------------------------------------------------------------------------
# GPU parity
# ---------------------------------------------------------------------------
def _cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from favor_random_feature_gb300 import build
    build.build()
    return torch


def _dev(torch, a, bf16):
    a = np.ascontiguousarray(a)
    if bf16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(a.astype(np.float32)).cuda()


def _run(inp, L0, T, fmap, use_f32=False):
    """State of the first L0 keys, then T decode steps (tokens L0 .. L0+T-1).
    Returns (state after the prefix as (S, z) float64, decode outputs
    [B][H][T][dv] float64)."""
    torch = _cuda()
    w = inp.w
    bf16 = w.dtype == "bf16" and not use_f32
    src_q, src_k, src_v = (inp.q, inp.k, inp.v) if bf16 else (inp.q32, inp.k32, inp.v32)
    m = w.d if fmap in NO_OMEGA else w.m
    r = fv.favor_feature_dim(fmap, w.d, m)
    per = fv.favor_state_floats(w.d, w.dv, m, fmap)
    om = None if fmap in NO_OMEGA else torch.from_numpy(
        np.ascontiguousarray(inp.omega, dtype=np.float32)).cuda()
    stream = torch.cuda.current_stream()
    state = torch.full((w.B, w.H, per), float("nan"), dtype=torch.float32, device="cuda")
    st_fn = fv.favor_attn_state if bf16 else fv.favor_attn_state_f32
    dec_fn = fv.favor_attn_decode if bf16 else fv.favor_attn_decode_f32
    kp = _dev(torch, src_k[:, :, :L0], bf16) if L0 else None
    vp = _dev(torch, src_v[:, :, :L0], bf16) if L0 else None
    rc = st_fn(kp, vp, om, state, w.B, w.H, L0, w.d, w.dv, m, fmap, stream)
    assert rc == fv.FAVOR_OK, fv.strerror(rc)
    s0 = state.cpu().numpy().astype(np.float64)
    outs = []
    for t in range(L0, L0 + T):
        q = _dev(torch, src_q[:, :, t], bf16)
        k = _dev(torch, src_k[:, :, t], bf16)
        v = _dev(torch, src_v[:, :, t], bf16)
        out = torch.full((w.B, w.H, w.dv), float("nan"), dtype=torch.float32, device="cuda")
        rc = dec_fn(q, k, v, om, state, out, w.B, w.H, w.d, w.dv, m, fmap, stream)
        assert rc == fv.FAVOR_OK, fv.strerror(rc)
        outs.append(out)
    st = fv.favor_get_device_status(stream)
    assert st == fv.FAVOR_OK, fv.strerror(st)
    got = torch.stack(outs, dim=2).cpu().numpy().astype(np.float64) if outs else None
    Sh = s0[..., : r * w.dv].reshape(w.B, w.H, r, w.dv)
    zh = s0[..., r * w.dv: r * (w.dv + 1)]
    rho = s0[..., r * (w.dv + 1):]
    return (Sh * np.exp2(rho)[..., None], zh * np.exp2(rho), rho), got


def _oracle_state(inp, L0, fmap):
    import oracle
    om = None if fmap in NO_OMEGA else inp.omega
    return oracle.state(inp.k32[:, :, :L0], inp.v32[:, :, :L0], om, feature_map=fmap)


def _state_err(got, ref):
    S, z, _ = got
    Sr, zr = ref
    a = np.concatenate([S, z[..., None]], axis=-1)
    b = np.concatenate([Sr, zr[..., None]], axis=-1)
    return (np.linalg.norm((a - b).reshape(a.shape[0], a.shape[1], -1), axis=-1) /
            np.linalg.norm(b.reshape(b.shape[0], b.shape[1], -1), axis=-1))


def _decode_ref(inp, L, fmap, heads=None):
    import oracle
    om = None if fmap in NO_OMEGA else inp.omega
    return oracle.forward(inp.q32[:, :, :L], inp.k32[:, :, :L], inp.v32[:, :, :L], om, causal=True,
                          feature_map=fmap, heads=heads)


CASES = [   # (workload, feature map, m or None, L0, T)
    (CAUSAL8K, MAP_POSITIVE, None, 300, 5),
    (CAUSAL8K.with_(dv=128), MAP_POSITIVE, None, 257, 3),
    (CAUSAL8K, MAP_TRIG, 128, 300, 4),
    (CAUSAL8K.with_(d=128, dv=32), MAP_ELU1, None, 200, 4),
    (LONG64K, MAP_POSITIVE, 768, 130, 3),        # r > 512: 128-feature tiles
    (CAUSAL8K, MAP_TRIG, 256, 129, 3),           # r = 512: a cluster of 8
    (CAUSAL8K, MAP_RELU, None, 200, 4),
    (CAUSAL8K.with_(omega="iid"), MAP_TRIG_SOFTMAX, 64, 150, 3),
    (CAUSAL8K, MAP_POSITIVE, 64, 200, 3),         # r = 64: one 64-feature tile
    (CAUSAL8K, MAP_ELU1, None, 200, 3),           # r = d = 64
]


@pytest.mark.gpu
@pytest.mark.parametrize("w,fmap,m,L0,T", CASES,
                         ids=["pos", "pos_dv128", "trig_r256", "elu_d128", "pos_r768", "trig_r512", "relu",
                              "trig_softmax", "pos_r64", "elu_d64"])
@pytest.mark.parametrize("f32", [False, True], ids=["bf16", "f32"])
def test_state_then_decode(w, fmap, m, L0, T, f32):
    w = w.with_(feature_map=fmap, **({"m": m} if m else {}))
    if fmap in NO_OMEGA:
        w = w.with_(m=w.d, omega="iid")
    inp = make_inputs(w, L=L0 + T, B=2, H=3)
    got_state, got = _run(inp, L0, T, fmap, use_f32=f32)
    es = _state_err(got_state, _oracle_state(inp, L0, fmap))
    assert es.max() <= (STATE_F32 if f32 else STATE_BF16), es.max()
    assert np.isfinite(got_state[2]).all()
    ref = _decode_ref(inp, L0 + T, fmap)[:, :, L0:]
    if fmap in (MAP_TRIG, MAP_TRIG_SOFTMAX):
        # trig denominators are not bounded away from zero (after a few
        # hundred keys every row is ill conditioned): the error of each row
        # is taken relative to its condition number, as for the forward pass
        from parity_util import causal_trig_condition, conditioned_errors
        kappa = causal_trig_condition(inp, fmap=fmap)[:, :, L0:]
        e = conditioned_errors(got, ref, kappa, inp.v32)
    else:
        e = row_errors(got, ref)
    if f32:
        assert e.max() <= F32_MAX, e.max()
    else:
        assert e.max() <= BF16_MAX and e.mean() <= BF16_MEAN, (e.max(), e.mean())


@pytest.mark.gpu
@pytest.mark.parametrize("fmap", [MAP_POSITIVE, MAP_TRIG, MAP_ELU1])
def test_decode_from_empty_state(fmap):
    """L0 = 0: the empty state, then the first tokens; out_0 = v_0 exactly
    for the positive map (one key)."""
    w = DEMO64.with_(feature_map=fmap, m=32 if fmap == MAP_ELU1 else 64, omega="iid")
    inp = make_inputs(w, L=12, B=1, H=2)
    st, got = _run(inp, 0, 12, fmap, use_f32=True)
    assert np.all(st[0] == 0) and np.all(st[1] == 0) and np.all(np.isneginf(st[2]))
    ref = _decode_ref(inp, 12, fmap)
    e = row_errors(got, ref)
    assert e.max() <= F32_MAX, e.max()


@pytest.mark.gpu
def test_decode_full_size_after_8192_tokens():
    """The benchmark shape: B=4, H=16, d=dv=64, m=256, the state of 8192
    keys, then 4 decode steps; two sampled heads against the oracle."""
    w = CAUSAL8K
    L0, T = 8192, 4
    inp = make_inputs(w, L=L0 + T)
    got_state, got = _run(inp, L0, T, MAP_POSITIVE)
    heads = [5, 58]
    ref = _decode_ref(inp, L0 + T, MAP_POSITIVE, heads=heads)[:, :, L0:]
    flat_g = got.reshape(w.B * w.H, T, w.dv)[heads]
    flat_r = ref.reshape(w.B * w.H, T, w.dv)[heads]
    e = row_errors(flat_g, flat_r)
    assert e.max() <= BF16_MAX and e.mean() <= BF16_MEAN, (e.max(), e.mean())
    # every head's state is finite and its z positive
    assert np.isfinite(got_state[0]).all() and (got_state[1] > 0).all()


@pytest.mark.gpu
def test_decode_steps_match_forward_rows():
    """Decoding every token of a sequence from the empty state gives the
    causal forward pass's rows (both through the library, fp32)."""
    torch = _cuda()
    from parity_util import run_gpu
    w = DEMO64.with_(m=128, omega="iid")
    inp = make_inputs(w, L=40, B=2, H=2)
    _, got = _run(inp, 0, 40, MAP_POSITIVE, use_f32=True)
    fwd = run_gpu(inp, True, MAP_POSITIVE)
    e = row_errors(got, fwd)
    assert e.max() <= F32_MAX, e.max()
    del torch
