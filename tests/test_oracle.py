"""Pins for the float64 oracle: each test ties it to something other than
itself -- a table the pages print, a closed form, brute force on tiny inputs,
a Monte-Carlo statement the pages make, or an invariant of the definition.
CPU only."""
import math
import os

import numpy as np
import pytest

import oracle
from favor_inputs import (CAUSAL8K, DEMO64, MAP_ELU1, MAP_POSITIVE, MAP_RELU, MAP_TRIG, MAP_TRIG_SOFTMAX,
                          bf16_bits, bf16_to_f32, make_inputs,
                          omega_block_orthogonal, omega_iid)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# independent closed forms used by the pins (not the oracle's code path)
# ---------------------------------------------------------------------------
def kernel_positive_closed(q, k, om):
    """(1/m) sum_i exp(w_i.(q+k) - (|q|^2+|k|^2)/2): the product of two
    positive features written as one sum, exp(-(|q|^2 + |k|^2)/2) times the
    mean of exp(w_i.(q + k)) (Performer page, the phi(x) equation)."""
    m = om.shape[0]
    s = om @ (q + k)
    return np.sum(np.exp(s - (q @ q + k @ k) / 2.0)) / m


def kernel_trig_closed(q, k, om):
    """(1/m) sum_i cos(w_i.(q-k)): sin a sin b + cos a cos b = cos(a-b)."""
    m = om.shape[0]
    return np.sum(np.cos(om @ (q - k))) / m


def brute_attention(Amat, V, causal):
    """O(L^2) attention with an explicit kernel matrix A_ij; lower triangle
    (diagonal included) when causal."""
    if causal:
        Amat = np.tril(Amat)
    return (Amat @ V) / (Amat @ np.ones(Amat.shape[1]))[:, None]


def softmax_attention(Q, K, V, scale):
    S = (Q @ K.T) * scale
    S = S - S.max(axis=1, keepdims=True)
    P = np.exp(S)
    P /= P.sum(axis=1, keepdims=True)
    return P @ V


# ---------------------------------------------------------------------------
# golden: the printed demo table of the Performer page, Out[27]
# ---------------------------------------------------------------------------
def test_page_demo_table_reproduced():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "performer_page_demo_table.txt"))
            if l.strip() and not l.startswith("#")]
    inp = make_inputs(DEMO64)
    Q = inp.q32[0, 0].astype(np.float64)
    K = inp.k32[0, 0].astype(np.float64)
    V = inp.v32[0, 0].astype(np.float64)
    n, d = Q.shape
    ref = softmax_attention(Q, K, V, 1.0 / math.sqrt(d))
    for m_s, cos_s, mse_s in rows:
        m = int(m_s)
        # the page's own projection: seed 0, randn(d, m) / sqrt(d)
        W = np.random.RandomState(0).randn(d, m) / np.sqrt(d)
        out = oracle.forward(Q[None, None], K[None, None], V[None, None], W.T[None],
                             causal=False)[0, 0]
        cos = np.mean([np.dot(ref[i], out[i]) / (np.linalg.norm(ref[i]) * np.linalg.norm(out[i]))
                       for i in range(n)])
        mse = np.mean((ref - out) ** 2)
        assert f"{cos:.4f}" == cos_s, (m, cos, cos_s)
        assert f"{mse:.6f}" == mse_s, (m, mse, mse_s)


# ---------------------------------------------------------------------------
# C1: closed form of phi(q)^T phi(k)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("d,m", [(32, 256), (64, 64), (128, 512)])
def test_positive_features_closed_form(d, m):
    rng = np.random.default_rng(7)
    om = rng.standard_normal((m, d))
    x = rng.standard_normal((6, d)) * d ** -0.25
    phi = oracle.features(x, om, MAP_POSITIVE)
    assert phi.shape == (6, m)
    for a in range(3):
        for b in range(3, 6):
            got = phi[a] @ phi[b]
            want = kernel_positive_closed(x[a], x[b], om)
            assert abs(got - want) <= 1e-13 * abs(want)


def test_trig_features_closed_form_and_order():
    rng = np.random.default_rng(8)
    d, m = 16, 64
    om = rng.standard_normal((m, d))
    x = rng.standard_normal((4, d)) * 0.5
    phi = oracle.features(x, om, MAP_TRIG)
    assert phi.shape == (4, 2 * m)
    # interleaved [sin(w1.x), cos(w1.x), ...] / sqrt(m), as printed
    p = om @ x[0]
    assert np.allclose(phi[0, 0::2] * math.sqrt(m), np.sin(p), rtol=0, atol=1e-14)
    assert np.allclose(phi[0, 1::2] * math.sqrt(m), np.cos(p), rtol=0, atol=1e-14)
    for a, b in [(0, 1), (2, 3), (1, 3)]:
        assert abs(phi[a] @ phi[b] - kernel_trig_closed(x[a], x[b], om)) <= 1e-14


def test_elu1_features_piecewise():
    x = np.array([[-2.0, -1e-300, 0.0, 1e-300, 0.5, 3.0]])
    phi = oracle.features(x, None, MAP_ELU1)
    # x+1 for x>0, e^x for x<=0; continuous at 0
    want = [math.exp(-2.0), 1.0, 1.0, 1.0, 1.5, 4.0]
    assert np.allclose(phi[0], want, rtol=1e-15, atol=0)


# ---------------------------------------------------------------------------
# C2 / C7: brute-force O(L^2) attention with the explicit kernel matrix
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("fmap", [MAP_POSITIVE, MAP_TRIG, MAP_ELU1, MAP_RELU, MAP_TRIG_SOFTMAX])
def test_bruteforce_kernel_attention(causal, fmap):
    rng = np.random.default_rng(11 + fmap)
    B, H, L, d, dv, m = 2, 2, 40, 16, 8, 32     # two batches of two heads: the [B][H] layout
    q = rng.standard_normal((B, H, L, d)) * d ** -0.25
    k = rng.standard_normal((B, H, L, d)) * d ** -0.25
    v = rng.standard_normal((B, H, L, dv))
    if fmap in (MAP_TRIG, MAP_TRIG_SOFTMAX):
        # small inputs keep the trig denominators well away from zero
        q *= 0.3
        k *= 0.3
    om = rng.standard_normal((H, m, d)) if fmap not in (MAP_ELU1, MAP_RELU) else None
    out = oracle.forward(q, k, v, om, causal=causal, feature_map=fmap)
    for b in range(B):
        for h in range(H):
            A = np.empty((L, L))
            for i in range(L):
                qi = q[b, h, i]
                for j in range(L):
                    kj = k[b, h, j]
                    if fmap == MAP_POSITIVE:
                        A[i, j] = kernel_positive_closed(qi, kj, om[h])
                    elif fmap == MAP_TRIG:
                        A[i, j] = kernel_trig_closed(qi, kj, om[h])
                    elif fmap == MAP_TRIG_SOFTMAX:
                        A[i, j] = math.exp((qi @ qi + kj @ kj) / 2) * kernel_trig_closed(qi, kj, om[h])
                    elif fmap == MAP_RELU:
                        A[i, j] = np.maximum(qi, 0) @ np.maximum(kj, 0)
                    else:
                        fq = np.where(qi > 0, qi + 1.0, np.exp(qi))
                        fk = np.where(kj > 0, kj + 1.0, np.exp(kj))
                        A[i, j] = fq @ fk
            ref = brute_attention(A, v[b, h], causal)
            err = np.max(np.abs(out[b, h] - ref)) / np.max(np.abs(ref))
            assert err <= 1e-12, (b, h, err)


def test_causal_reduces_to_noncausal_at_last_row_and_v0_at_first():
    inp = make_inputs(CAUSAL8K, L=50, B=1, H=2)
    args = (inp.q32, inp.k32, inp.v32, inp.omega)
    oc = oracle.forward(*args, causal=True)
    on = oracle.forward(*args, causal=False)
    assert np.allclose(oc[:, :, -1], on[:, :, -1], rtol=1e-13, atol=1e-15)
    # row 0 attends only to key 0: out_0 = v_0 (up to one rounding)
    assert np.allclose(oc[:, :, 0], inp.v32[:, :, 0], rtol=1e-14, atol=1e-15)


# ---------------------------------------------------------------------------
# C3: Monte-Carlo unbiasedness and O(1/m) variance (pages: E[phi(q)^T phi(k)]
# = exp(q^T k); "variance decreases as O(1/m)")
# ---------------------------------------------------------------------------
def _mc_estimates(q, k, m, T, seed, fmap=MAP_POSITIVE, orth=False):
    rng = np.random.default_rng(seed)
    d = q.shape[0]
    x = np.stack([q, k])
    est = np.empty(T)
    for t in range(T):
        if orth:
            om = omega_block_orthogonal(rng, 1, m, d)[0].astype(np.float64)
        else:
            om = rng.standard_normal((m, d))
        phi = oracle.features(x, om, fmap)
        est[t] = phi[0] @ phi[1]
    return est


def _qk_pair(d, seed, scale):
    rng = np.random.default_rng(seed)
    return rng.standard_normal(d) * scale, rng.standard_normal(d) * scale


def test_monte_carlo_unbiased_and_variance_1_over_m():
    d = 8
    q, k = _qk_pair(d, 3, 0.25)
    target = math.exp(q @ k)
    var1 = math.exp(2 * q @ k) * (math.exp((q + k) @ (q + k)) - 1.0)  # one feature
    T = 3000
    ms = [16, 32, 64, 128, 256]
    variances = []
    for i, m in enumerate(ms):
        est = _mc_estimates(q, k, m, T, 100 + i)
        se = math.sqrt(var1 / m / T)
        assert abs(est.mean() - target) <= 5 * se, (m, est.mean(), target, se)
        s2 = est.var(ddof=1)
        assert abs(s2 / (var1 / m) - 1.0) < 0.2, (m, s2, var1 / m)
        variances.append(s2)
    slope = np.polyfit(np.log(ms), np.log(variances), 1)[0]
    assert abs(slope + 1.0) < 0.1, slope


def test_monte_carlo_orthogonal_unbiased_and_not_worse():
    d = 8
    q, k = _qk_pair(d, 5, 0.25)
    target = math.exp(q @ k)
    var1 = math.exp(2 * q @ k) * (math.exp((q + k) @ (q + k)) - 1.0)
    m, T = 16, 3000
    est_o = _mc_estimates(q, k, m, T, 7, orth=True)
    est_i = _mc_estimates(q, k, m, T, 8, orth=False)
    se = math.sqrt(var1 / m / T)
    assert abs(est_o.mean() - target) <= 5 * se
    # orthogonal rows: variance no larger than iid (soft, 20% slack)
    assert est_o.var() <= 1.2 * est_i.var()


def test_monte_carlo_trig_gaussian_kernel():
    d = 8
    q, k = _qk_pair(d, 9, 0.3)
    dl = (q - k) @ (q - k)
    target = math.exp(-dl / 2)
    var1 = (1 + math.exp(-2 * dl)) / 2 - math.exp(-dl)
    m, T = 32, 3000
    est = _mc_estimates(q, k, m, T, 10, fmap=MAP_TRIG)
    se = math.sqrt(var1 / m / T)
    assert abs(est.mean() - target) <= 5 * se
    assert abs(est.var(ddof=1) / (var1 / m) - 1.0) < 0.2


# ---------------------------------------------------------------------------
# C6: textbook limit -- large m approaches exact softmax attention exp(q^T k)
# ---------------------------------------------------------------------------
def test_large_m_approaches_softmax_attention():
    rng = np.random.default_rng(21)
    L, d, dv = 12, 8, 4
    # |q+k|^2 ~ 2: the per-feature variance factor exp(|q+k|^2)-1 stays small
    q = rng.standard_normal((L, d)) * 0.35
    k = rng.standard_normal((L, d)) * 0.35
    v = rng.standard_normal((L, dv))
    ref = softmax_attention(q, k, v, 1.0)      # logits q^T k, inputs pre-scaled
    errs = {}
    for m in (256, 65536):
        om = rng.standard_normal((1, m, d))
        out = oracle.forward(q[None, None], k[None, None], v[None, None], om, causal=False)[0, 0]
        errs[m] = np.max(np.abs(out - ref))
    assert errs[65536] < 0.02
    assert errs[65536] < errs[256] / 4


# ---------------------------------------------------------------------------
# C4 / C5: positivity and invariances
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("fmap", [MAP_POSITIVE, MAP_ELU1])
def test_features_and_denominators_positive(fmap):
    inp = make_inputs(CAUSAL8K, L=64, B=1, H=2)
    om = inp.omega if fmap == MAP_POSITIVE else None
    for h in range(2):
        phi = oracle.features(inp.q32[0, h], om[h] if om is not None else None, fmap)
        assert np.all(phi > 0)
    for causal in (False, True):
        out, den = oracle.forward(inp.q32, inp.k32, inp.v32, om, causal=causal,
                                  feature_map=fmap, return_den=True)
        assert np.all(den > 0)
        # a convex combination of the v rows: inside their column range
        vmin = inp.v32.min(axis=2, keepdims=True)
        vmax = inp.v32.max(axis=2, keepdims=True)
        assert np.all(out >= vmin - 1e-12) and np.all(out <= vmax + 1e-12)


def test_constant_values_reproduced():
    inp = make_inputs(CAUSAL8K, L=30, B=1, H=1)
    v = np.broadcast_to(np.arange(64.0)[None, None, None, :] - 20.0, inp.v32.shape)
    for causal in (False, True):
        out = oracle.forward(inp.q32, inp.k32, v, inp.omega, causal=causal)
        assert np.allclose(out, v, rtol=1e-13, atol=1e-12)


@pytest.mark.parametrize("fmap", [MAP_POSITIVE, MAP_ELU1, MAP_TRIG], ids=["positive", "elu1", "trig"])
def test_zero_keys_give_the_mean_of_the_values(fmap):
    """Every key zero: phi(0) is the same vector for every key (1/sqrt(m) for
    the positive map, ones for ELU+1, [0, 1, 0, 1, ...]/sqrt(m) for sin/cos),
    so each query weighs the keys it sees equally whatever q and omega are:
    out_i = mean of v_0..v_i (causal), the mean of all v (non-causal)."""
    w = CAUSAL8K.with_(feature_map=fmap, m=64 if fmap == MAP_ELU1 else 256)
    inp = make_inputs(w, L=50, B=1, H=2)
    q = inp.q32 * (0.25 if fmap == MAP_TRIG else 1.0)   # sin/cos: keep sum_i cos(w_i.q) away from 0
    k = np.zeros_like(inp.k32)
    v = inp.v32.astype(np.float64)
    om = None if fmap == MAP_ELU1 else inp.omega
    want_c = np.cumsum(v, axis=2) / np.arange(1, v.shape[2] + 1)[:, None]
    want_n = np.broadcast_to(v.mean(axis=2, keepdims=True), v.shape)
    assert np.allclose(oracle.forward(q, k, inp.v32, om, causal=True, feature_map=fmap), want_c,
                       rtol=1e-11, atol=1e-12)
    assert np.allclose(oracle.forward(q, k, inp.v32, om, causal=False, feature_map=fmap), want_n,
                       rtol=1e-11, atol=1e-12)


def test_permuting_omega_rows_is_invariant():
    inp = make_inputs(CAUSAL8K, L=33, B=1, H=1)
    perm = np.random.default_rng(0).permutation(inp.omega.shape[1])
    for causal in (False, True):
        a = oracle.forward(inp.q32, inp.k32, inp.v32, inp.omega, causal=causal)
        b = oracle.forward(inp.q32, inp.k32, inp.v32, inp.omega[:, perm], causal=causal)
        assert np.allclose(a, b, rtol=1e-12, atol=1e-13)


def test_head_subset_matches_full():
    inp = make_inputs(CAUSAL8K, L=20, B=2, H=3)
    full = oracle.forward(inp.q32, inp.k32, inp.v32, inp.omega, causal=True)
    sub = oracle.forward(inp.q32, inp.k32, inp.v32, inp.omega, causal=True, heads=[4, 1])
    flat_f = full.reshape(6, 20, 64)
    flat_s = sub.reshape(6, 20, 64)
    assert np.array_equal(flat_f[[1, 4]], flat_s[[1, 4]])
    assert np.isnan(flat_s[0]).all()


# ---------------------------------------------------------------------------
# the input generators: bf16 rounding and block-orthogonal omega
# ---------------------------------------------------------------------------
def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    x = np.random.default_rng(0).standard_normal(100000).astype(np.float32) * 7
    x[:4] = [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8, 0.0]   # ties
    got = bf16_bits(x)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)
    back = bf16_to_f32(got)
    assert np.all(np.abs(back - x) <= np.abs(x) * 2.0 ** -8)


def test_block_orthogonal_omega():
    from scipy import stats
    rng = np.random.default_rng(3)
    d, m = 16, 40
    om = omega_block_orthogonal(rng, 50, m, d).astype(np.float64)
    for h in range(3):
        for b0, b1 in [(0, 16), (16, 32), (32, 40)]:
            blk = om[h, b0:b1]
            n = blk / np.linalg.norm(blk, axis=1, keepdims=True)
            g = n @ n.T
            assert np.allclose(g, np.eye(b1 - b0), atol=1e-6)   # fp32 storage
    # row lengths ~ chi(d)
    lengths = np.linalg.norm(om.reshape(-1, d), axis=1)
    assert stats.kstest(lengths, stats.chi(d).cdf).pvalue > 1e-3
    # iid draws are N(0,1) entries
    iid = omega_iid(rng, 4, 64, d).ravel()
    assert stats.kstest(iid, "norm").pvalue > 1e-3


# ---------------------------------------------------------------------------
# C5 (i): a positive factor per query row and one per head on the keys leave
# the output unchanged (what the GPU stabilisers rely on).  Brute force with
# the query norm term and 1/m dropped and the keys scaled by 7.3 must equal
# the oracle.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
def test_row_and_head_scaling_invariance(causal):
    rs = np.random.default_rng(11)
    L, d, m = 40, 16, 64
    q = rs.standard_normal((L, d)) * 0.4
    k = rs.standard_normal((L, d)) * 0.4
    v = rs.standard_normal((L, 8))
    om = omega_iid(np.random.default_rng(12), 1, m, d)[0]
    fq = np.exp(q @ om.T)                                   # no -|q|^2/2, no 1/sqrt(m)
    fk = 7.3 * np.exp(k @ om.T - 0.5 * np.sum(k * k, axis=1, keepdims=True))
    want = brute_attention(fq @ fk.T, v, causal)
    got = oracle.forward(q[None, None], k[None, None], v[None, None], om[None], causal=causal,
                         feature_map=MAP_POSITIVE)[0, 0]
    assert np.allclose(got, want, rtol=1e-11, atol=1e-13)


# ---------------------------------------------------------------------------
# C5 (v): with positive features every output is a convex combination of the
# value rows it attends to, so each column lies within their range
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("fmap", [MAP_POSITIVE, MAP_ELU1])
def test_outputs_within_value_range(causal, fmap):
    rs = np.random.default_rng(13)
    L, d = 50, 16
    m = d if fmap == MAP_ELU1 else 48
    q = rs.standard_normal((1, 1, L, d)) * 0.5
    k = rs.standard_normal((1, 1, L, d)) * 0.5
    v = rs.standard_normal((1, 1, L, 6))
    om = None if fmap == MAP_ELU1 else omega_iid(np.random.default_rng(14), 1, m, d)
    out = oracle.forward(q, k, v, om, causal=causal, feature_map=fmap)[0, 0]
    vv = v[0, 0]
    for i in range(L):
        seen = vv[: i + 1] if causal else vv
        assert np.all(out[i] >= seen.min(axis=0) - 1e-12) and np.all(out[i] <= seen.max(axis=0) + 1e-12)


# ---------------------------------------------------------------------------
# carried state and the one-token decode step (study notes, "Case 2": the
# running sums S_i, z_i)
# ---------------------------------------------------------------------------
def _features_numpy(x, om, fmap):
    """Closed-form features written out in numpy: positive exp(w.x - |x|^2/2)/sqrt(m),
    trig (sin, cos) pairs interleaved per projection over sqrt(m), elu1 elementwise."""
    if fmap == MAP_ELU1:
        return np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))
    m = om.shape[0]
    p = x @ om.T
    if fmap == MAP_POSITIVE:
        return np.exp(p - 0.5 * np.sum(x * x, axis=1, keepdims=True)) / math.sqrt(m)
    out = np.empty((x.shape[0], 2 * m))
    out[:, 0::2], out[:, 1::2] = np.sin(p), np.cos(p)
    return out / math.sqrt(m)


def _kernel_matrix(q, k, om, fmap):
    """A_ij = phi(q_i).phi(k_j) by the single-sum closed forms (positive, trig)
    or the elementwise product (elu1) -- no feature vectors formed."""
    if fmap == MAP_POSITIVE:
        return np.array([[kernel_positive_closed(a, b, om) for b in k] for a in q])
    if fmap == MAP_TRIG:
        return np.array([[kernel_trig_closed(a, b, om) for b in k] for a in q])
    e = lambda x: np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))
    return e(q) @ e(k).T


def _small_head(seed, L, d, dv, m, fmap, scale=0.4):
    rs = np.random.default_rng(seed)
    q = rs.standard_normal((1, 2, L, d)) * scale
    k = rs.standard_normal((1, 2, L, d)) * scale
    v = rs.standard_normal((1, 2, L, dv))
    om = None if fmap == MAP_ELU1 else omega_iid(np.random.default_rng(seed + 1), 2, m, d)
    return q, k, v, om


@pytest.mark.parametrize("fmap", [MAP_POSITIVE, MAP_TRIG, MAP_ELU1])
def test_state_matches_closed_form_features(fmap):
    q, k, v, om = _small_head(21, 30, 16, 8, 24, fmap)
    S, z = oracle.state(k, v, om, feature_map=fmap)
    for h in range(2):
        phi = _features_numpy(k[0, h], None if om is None else om[h], fmap)
        assert np.allclose(S[0, h], phi.T @ v[0, h], rtol=1e-12, atol=1e-14)
        assert np.allclose(z[0, h], phi.sum(axis=0), rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("fmap", [MAP_POSITIVE, MAP_TRIG, MAP_ELU1])
def test_decode_steps_from_empty_state_are_brute_causal(fmap):
    L, d, dv, m = 12, 8, 5, 16
    q, k, v, om = _small_head(23, L, d, dv, m, fmap)
    r = oracle.feature_dim(fmap, d, m)
    S, z = np.zeros((1, 2, r, dv)), np.zeros((1, 2, r))
    outs = []
    for t in range(L):
        o, S, z = oracle.decode_step(q[:, :, t], k[:, :, t], v[:, :, t], om, S, z, feature_map=fmap)
        outs.append(o)
    got = np.stack(outs, axis=2)
    for h in range(2):
        A = _kernel_matrix(q[0, h], k[0, h], None if om is None else om[h], fmap)
        want = brute_attention(A, v[0, h], causal=True)
        assert np.allclose(got[0, h], want, rtol=1e-9, atol=1e-11)


def test_state_is_additive_and_decode_continues_a_prefix():
    L, a = 40, 27
    q, k, v, om = _small_head(25, L, 16, 8, 32, MAP_POSITIVE)
    S, z = oracle.state(k, v, om)
    S1, z1 = oracle.state(k[:, :, :a], v[:, :, :a], om)
    S2, z2 = oracle.state(k[:, :, a:], v[:, :, a:], om)
    assert np.allclose(S1 + S2, S, rtol=1e-12, atol=1e-14) and np.allclose(z1 + z2, z, rtol=1e-12)
    # decoding tokens a.. from the state of the first a keys gives the causal rows a..
    full = oracle.forward(q, k, v, om, causal=True)
    St, zt = S1, z1
    for t in range(a, L):
        o, St, zt = oracle.decode_step(q[:, :, t], k[:, :, t], v[:, :, t], om, St, zt)
        assert np.allclose(o, full[:, :, t], rtol=1e-11, atol=1e-13)
    assert np.allclose(St, S, rtol=1e-11) and np.allclose(zt, z, rtol=1e-11)


# ---------------------------------------------------------------------------
# random projections drawn by a counter-based generator: Philox4x64-10
# (Salmon et al., SC 2011) against numpy's implementation of the same
# generator, Box-Muller normals by their distribution, and the
# block-orthogonal rows against a QR factorisation and the chi law of norms
# ---------------------------------------------------------------------------
def _numpy_philox_block(counter, key):
    """numpy advances its counter before a block: start it one below."""
    c = sum(int(x) << (64 * i) for i, x in enumerate(counter))
    c = (c - 1) % (1 << 256)
    words = np.array([(c >> (64 * i)) & ((1 << 64) - 1) for i in range(4)], dtype=np.uint64)
    g = np.random.Philox(key=np.array(key, dtype=np.uint64), counter=words)
    return [int(x) for x in g.random_raw(4)]


@pytest.mark.parametrize("counter,key", [
    ([0, 0, 0, 0], [0, 0]),
    ([1, 0, 0, 0], [5, 7]),
    ([0, 1, 0, 0], [2**64 - 1, 3]),                        # a carry into the second word
    ([2**64 - 1, 2**64 - 1, 0, 9], [123456789, 987654321]),
    ([12345, 0, 1, 0], [2024, 0]),                         # the stream word of the draws
])
def test_philox_matches_numpy(counter, key):
    assert oracle.philox4x64(counter, key) == _numpy_philox_block(counter, key)


def test_normals_are_standard_and_streams_independent():
    from scipy import stats
    n = 100_000
    z0 = np.array([oracle.normal(7, 0, e) for e in range(n)])
    z1 = np.array([oracle.normal(7, 1, e) for e in range(n)])
    for z in (z0, z1):
        assert stats.kstest(z, "norm").pvalue > 1e-3
        assert abs(z.mean()) < 5 / np.sqrt(n) and abs(z.var() - 1) < 5 * np.sqrt(2 / n)
    assert abs(np.corrcoef(z0, z1)[0, 1]) < 5 / np.sqrt(n)
    assert abs(np.corrcoef(z0[:-1], z0[1:])[0, 1]) < 5 / np.sqrt(n)
    assert oracle.normal(8, 0, 0) != oracle.normal(7, 0, 0)


def test_draw_omega_iid_is_the_normal_stream():
    from scipy import stats
    w = oracle.draw_omega(3, 40, 32, 0, 99)
    flat = w.reshape(-1)
    assert all(flat[e] == oracle.normal(99, 0, e) for e in range(0, flat.size, 97))
    assert stats.kstest(flat, "norm").pvalue > 1e-3


@pytest.mark.parametrize("m,d", [(64, 32), (100, 32), (256, 64)])
def test_draw_omega_block_orthogonal(m, d):
    """Each block's rows are the orthonormal factor of its Gaussian block (QR
    of the transpose with a positive diagonal) scaled by chi(d) norms drawn
    from the second stream; the last block is truncated to m rows."""
    from scipy import stats
    H, seed = 2, 31
    w = oracle.draw_omega(H, m, d, 1, seed)
    nb = -(-m // d)
    norms = []
    for h in range(H):
        for b in range(nb):
            base = (h * nb + b) * d * d
            G = np.array([oracle.normal(seed, 0, base + i) for i in range(d * d)]).reshape(d, d)
            Q, R = np.linalg.qr(G.T)
            Q = Q * np.sign(np.diag(R))
            rows = min(d, m - b * d)
            chi = np.array([np.linalg.norm([oracle.normal(seed, 1, base + i * d + t) for t in range(d)])
                            for i in range(rows)])
            want = Q.T[:rows] * chi[:, None]
            got = w[h, b * d: b * d + rows]
            assert np.allclose(got, want, rtol=1e-10, atol=1e-10)
            gram = got @ got.T
            assert np.allclose(gram - np.diag(np.diag(gram)), 0, atol=1e-10 * d)
            norms.extend(np.linalg.norm(got, axis=1))
    if len(norms) >= 100:
        assert stats.kstest(norms, stats.chi(d).cdf).pvalue > 1e-3


# ---------------------------------------------------------------------------
# ReLU ("Kernel Feature Maps" section 2) and the softmax-scaled Fourier map
# (section 3's additional scaling)
# ---------------------------------------------------------------------------
def test_relu_features_and_homogeneity():
    x = np.array([[-1.5, 0.0, 0.25, 3.0]])
    assert np.array_equal(oracle.features(x, None, MAP_RELU), [[0.0, 0.0, 0.25, 3.0]])
    # phi(c x) = c phi(x) for c > 0: scaling queries or keys leaves the output unchanged
    rng = np.random.default_rng(41)
    q, k = rng.standard_normal((1, 1, 30, 16)), rng.standard_normal((1, 1, 30, 16))
    v = rng.standard_normal((1, 1, 30, 4))
    for causal in (False, True):
        a = oracle.forward(q, k, v, None, causal=causal, feature_map=MAP_RELU)
        b = oracle.forward(2.5 * q, 0.5 * k, v, None, causal=causal, feature_map=MAP_RELU)
        assert np.allclose(a, b, rtol=1e-12, atol=1e-14)


def test_trig_softmax_closed_form_and_monte_carlo_softmax_kernel():
    d, m = 8, 16
    q, k = _qk_pair(d, 13, 0.25)
    om = np.random.default_rng(14).standard_normal((m, d))
    phi = oracle.features(np.stack([q, k]), om, MAP_TRIG_SOFTMAX)
    closed = math.exp((q @ q + k @ k) / 2) * kernel_trig_closed(q, k, om)
    assert abs(phi[0] @ phi[1] - closed) <= 1e-13 * abs(closed)
    # unbiased for the softmax kernel exp(q.k): E = exp(|q|^2/2 + |k|^2/2) exp(-|q-k|^2/2);
    # one feature pair's variance is that of the Gaussian-kernel estimate times exp(|q|^2+|k|^2)
    T = 4000
    est = _mc_estimates(q, k, m, T, 15, fmap=MAP_TRIG_SOFTMAX)
    dl = (q - k) @ (q - k)
    var1 = math.exp(q @ q + k @ k) * ((1 + math.exp(-2 * dl)) / 2 - math.exp(-dl))
    se = math.sqrt(var1 / m / T)
    assert abs(est.mean() - math.exp(q @ k)) <= 5 * se, (est.mean(), math.exp(q @ k), se)
    assert abs(est.var(ddof=1) / (var1 / m) - 1.0) < 0.2


# ---------------------------------------------------------------------------
# backward pass: central finite differences of the forward pass (float64) on
# sampled entries of every input, for every map, causal and not
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("fmap", [MAP_POSITIVE, MAP_TRIG, MAP_ELU1, MAP_RELU, MAP_TRIG_SOFTMAX])
def test_backward_matches_finite_differences(causal, fmap):
    rs = np.random.default_rng(51 + fmap)
    B, H, L, d, dv, m = 2, 2, 9, 8, 5, 12
    scale = 0.3 if fmap in (MAP_TRIG, MAP_TRIG_SOFTMAX) else 0.5
    q = rs.standard_normal((B, H, L, d)) * scale
    k = rs.standard_normal((B, H, L, d)) * scale
    if fmap == MAP_RELU:
        # keep every query's features in touch with some key mass, and away
        # from the kink at 0 where the derivative jumps
        q, k = np.abs(q) + 0.05, np.abs(k) + 0.05
        q[..., ::3] *= -1
    v = rs.standard_normal((B, H, L, dv))
    g = rs.standard_normal((B, H, L, dv))
    om = None if fmap in (MAP_ELU1, MAP_RELU) else rs.standard_normal((H, m, d))
    dq, dk, dv_, dw = oracle.backward(q, k, v, om, g, causal, fmap)

    def loss(q_, k_, v_, om_):
        return float(np.sum(oracle.forward(q_, k_, v_, om_, causal=causal, feature_map=fmap) * g))

    h = 1e-6
    tensors = [("q", q, dq), ("k", k, dk), ("v", v, dv_)] + ([("w", om, dw)] if om is not None else [])
    for name, arr, grad in tensors:
        for _ in range(6):
            idx = tuple(int(rs.integers(0, n)) for n in arr.shape)
            a, b = arr.copy(), arr.copy()
            a[idx] += h
            b[idx] -= h
            sub = {"q": 0, "k": 1, "v": 2, "w": 3}[name]
            args_a, args_b = [q, k, v, om], [q, k, v, om]
            args_a[sub], args_b[sub] = a, b
            fd = (loss(*args_a) - loss(*args_b)) / (2 * h)
            assert abs(fd - grad[idx]) <= 1e-6 * (abs(grad[idx]) + np.abs(grad).max()), (name, idx, fd, grad[idx])


def test_backward_single_token_passes_the_gradient_to_v():
    """L = 1: out = v exactly, so dv = g and dq = dk = dw = 0."""
    rs = np.random.default_rng(61)
    q, k = rs.standard_normal((1, 2, 1, 8)), rs.standard_normal((1, 2, 1, 8))
    v, g = rs.standard_normal((1, 2, 1, 4)), rs.standard_normal((1, 2, 1, 4))
    om = rs.standard_normal((2, 16, 8))
    for causal in (False, True):
        dq, dk, dv, dw = oracle.backward(q, k, v, om, g, causal)
        assert np.allclose(dv, g, rtol=1e-13, atol=1e-15)
        assert np.abs(dq).max() < 1e-12 and np.abs(dk).max() < 1e-12 and np.abs(dw).max() < 1e-12
