"""How sharp the GPU parity bar is.  The bf16 bar (per-row normwise error
e_i = |o_i - ref_i| / |ref_i|, max <= 2e-2 and mean <= 2e-3) must reject the
plausible bugs of a chunked, stabilised, split kernel and admit the
kernels' own operand precision.  Each bug is emulated here in float64 on the
CPU, from the oracle's features, on a reduced causal8k / nc4096 shape
(block-orthogonal omega, bf16-rounded inputs), and compared with the oracle
through the same metric the GPU parity tests use."""
import numpy as np
import pytest

import oracle
from favor_inputs import CAUSAL8K, NC4096, bf16_bits, bf16_to_f32, make_inputs
from parity_util import row_errors

L, H = 1024, 2      # causal case: 8 chunks of 128 rows per head
LN = 1536           # non-causal case: 3 pieces of 512 keys per head
MAX_BAR, MEAN_BAR = 2e-2, 2e-3


def passes(e):
    return e.max() <= MAX_BAR and e.mean() <= MEAN_BAR


@pytest.fixture(scope="module")
def causal():
    inp = make_inputs(CAUSAL8K, L=L, B=1, H=H)
    ref = oracle.forward(inp.q32, inp.k32, inp.v32, inp.omega, causal=True)
    feats = [(oracle.features(inp.q32[0, h], inp.omega[h]), oracle.features(inp.k32[0, h], inp.omega[h]))
             for h in range(H)]
    return inp, ref, feats


@pytest.fixture(scope="module")
def noncausal():
    inp = make_inputs(NC4096, L=LN, B=1, H=H)
    ref = oracle.forward(inp.q32, inp.k32, inp.v32, inp.omega, causal=False)
    return inp, ref


def weighted(causal, weight):
    """out_i = sum_j W_ij A_ij v_j / sum_j W_ij A_ij with A_ij = phi(q_i).phi(k_j):
    the causal form is W = [j <= i]; a bug changes W."""
    inp, ref, feats = causal
    out = np.empty_like(ref)
    i, j = np.arange(L)[:, None], np.arange(L)[None, :]
    W = weight(i, j)
    for h, (pq, pk) in enumerate(feats):
        A = (pq @ pk.T) * W
        with np.errstate(invalid="ignore", divide="ignore"):
            out[0, h] = (A @ inp.v32[0, h].astype(np.float64)) / A.sum(1, keepdims=True)
    return out


def test_control_brute_force_with_the_causal_mask_passes(causal):
    _, ref, _ = causal
    e = row_errors(weighted(causal, lambda i, j: (j <= i) * 1.0), ref)
    assert e.max() < 1e-12


def test_kernels_fp16_omega_is_admitted(causal):
    inp, ref, _ = causal
    om16 = inp.omega.astype(np.float16).astype(np.float32)
    assert passes(row_errors(oracle.forward(inp.q32, inp.k32, inp.v32, om16, causal=True), ref))


def test_bf16_omega_is_rejected(causal):
    inp, ref, _ = causal
    om = bf16_to_f32(bf16_bits(inp.omega)).reshape(inp.omega.shape)
    assert not passes(row_errors(oracle.forward(inp.q32, inp.k32, inp.v32, om, causal=True), ref))


CAUSAL_BUGS = {
    "diagonal left out": lambda i, j: (j < i) * 1.0,
    "chunk 3 missing from the state carried past it":
        lambda i, j: ((j <= i) & ~((j >= 384) & (j < 512) & (i >= 512))) * 1.0,
    "chunk 0 missing from every later chunk's state": lambda i, j: ((j <= i) & ~((j < 128) & (i >= 128))) * 1.0,
    "last key of each chunk left out of the carried state":
        lambda i, j: ((j <= i) & ~((j % 128 == 127) & (j // 128 < i // 128))) * 1.0,
    "first key of each chunk left out of the carried state":
        lambda i, j: ((j <= i) & ~((j % 128 == 0) & (j // 128 < i // 128))) * 1.0,
    "carried state entering chunk 4 off by a factor 2 (a missed power-of-two rescale)":
        lambda i, j: np.where((j < 512) & (i >= 512), 2.0, 1.0) * (j <= i),
    "carried state entering chunk 4 off by 10 %":
        lambda i, j: np.where((j < 512) & (i >= 512), 1.1, 1.0) * (j <= i),
}


@pytest.mark.parametrize("bug", list(CAUSAL_BUGS))
def test_causal_bug_is_rejected(causal, bug):
    _, ref, _ = causal
    out = weighted(causal, CAUSAL_BUGS[bug])
    rows = slice(1, None) if bug == "diagonal left out" else slice(None)   # row 0 is 0/0 there
    assert not passes(row_errors(out[:, :, rows], ref[:, :, rows])), bug


@pytest.mark.parametrize("lo,hi", [(0, 512), (1024, 1536), (1535, 1536)],
                         ids=["first piece", "last piece", "last key"])
def test_noncausal_keys_left_out_of_the_state_are_rejected(noncausal, lo, hi):
    inp, ref = noncausal
    keep = np.ones(LN, bool)
    keep[lo:hi] = False
    out = np.empty_like(ref)
    for h in range(H):
        pq = oracle.features(inp.q32[0, h], inp.omega[h])
        pk = oracle.features(inp.k32[0, h], inp.omega[h])[keep]
        out[0, h] = (pq @ (pk.T @ inp.v32[0, h][keep].astype(np.float64))) / (pq @ pk.sum(0))[:, None]
    assert not passes(row_errors(out, ref))


def test_fp32_bar_admits_fp32_features_and_rejects_fp16_omega():
    """The fp32 bar (max 1e-4) on the page's demo head (L = 64, d = 32, m = 256):
    features rounded to fp32 pass it; omega rounded to fp16 (the tensor-core
    operand precision) does not."""
    from favor_inputs import DEMO64
    inp = make_inputs(DEMO64)
    q, k, v, om = inp.q32[0, 0], inp.k32[0, 0], inp.v32[0, 0].astype(np.float64), inp.omega[0]
    ref = oracle.forward(inp.q32, inp.k32, inp.v32, inp.omega, causal=False)[0, 0]

    def out_from(pq, pk):
        return (pq @ (pk.T @ v)) / (pq @ pk.sum(0))[:, None]

    f32 = lambda a: a.astype(np.float32).astype(np.float64)
    e32 = row_errors(out_from(f32(oracle.features(q, om)), f32(oracle.features(k, om))), ref)
    assert e32.max() <= 1e-4
    om16 = om.astype(np.float16).astype(np.float32)
    e16 = row_errors(out_from(oracle.features(q, om16), oracle.features(k, om16)), ref)
    assert e16.max() > 1e-4


# ---------------------------------------------------------------------------
# the condition-normalised metric of the sin/cos map at the sweep shape
# (d = dv = 128, m = 256, causal): |o_i - ref_i| / (kappa_i (max_j |v_j| +
# |ref_i|)) must still reject a swapped sin/cos and a sign error
# ---------------------------------------------------------------------------
LT = 512


@pytest.fixture(scope="module")
def sweep_trig():
    from favor_inputs import MAP_TRIG, SWEEP16K
    from parity_util import causal_trig_condition
    w = SWEEP16K.with_(m=256, feature_map=MAP_TRIG)
    inp = make_inputs(w, L=LT, B=1, H=2)
    ref = oracle.forward(inp.q32, inp.k32, inp.v32, inp.omega, causal=True, feature_map=MAP_TRIG)
    kap = causal_trig_condition(inp)
    feats = [(oracle.features(inp.q32[0, h], inp.omega[h], MAP_TRIG),
              oracle.features(inp.k32[0, h], inp.omega[h], MAP_TRIG)) for h in range(H)]
    return inp, ref, kap, feats


def _trig_causal(inp, feats, tq=lambda p: p, tk=lambda p: p):
    out = np.empty((1, H, LT, inp.w.dv))
    mask = np.tril(np.ones((LT, LT)))
    for h, (pq, pk) in enumerate(feats):
        A = (tq(pq) @ tk(pk).T) * mask
        out[0, h] = (A @ inp.v32[0, h].astype(np.float64)) / A.sum(1, keepdims=True)
    return out


def _swap_sin_cos(p):
    s = p.copy()
    s[:, 0::2], s[:, 1::2] = p[:, 1::2], p[:, 0::2]
    return s


def _negate_sin(p):
    s = p.copy()
    s[:, 0::2] = -p[:, 0::2]
    return s


def _conditioned_passes(out, sweep):
    from parity_util import conditioned_errors
    inp, ref, kap, _ = sweep
    return passes(conditioned_errors(out, ref, kap, inp.v32))


def test_conditioned_metric_admits_the_exact_features(sweep_trig):
    inp, _, _, feats = sweep_trig
    assert _conditioned_passes(_trig_causal(inp, feats), sweep_trig)


@pytest.mark.parametrize("bug", ["queries' sin and cos swapped", "keys' sin negated",
                                 "keys' sin and cos swapped"])
def test_conditioned_metric_rejects_trig_bugs(sweep_trig, bug):
    inp, _, _, feats = sweep_trig
    if bug == "queries' sin and cos swapped":
        out = _trig_causal(inp, feats, tq=_swap_sin_cos)
    elif bug == "keys' sin negated":
        out = _trig_causal(inp, feats, tk=_negate_sin)
    else:
        out = _trig_causal(inp, feats, tk=_swap_sin_cos)
    assert not _conditioned_passes(out, sweep_trig), bug
