"""GPU parity: the CUDA path, called through the C ABI, against the float64
oracle on the same seeded inputs and the same omega.

Metric (per row): e_i = |o_i - ref_i|_2 / |ref_i|_2.
  fp32 inputs: max_i e_i <= 1e-4.
  bf16 inputs: max_i e_i <= 2e-2 and mean_i e_i <= 2e-3.
The sin/cos map has denominators that are not bounded away from zero: on
inputs where they are well conditioned (kappa <= 10) the plain metric
applies; on the sweep workload, where nearly every row is ill conditioned,
the error is normalised by each row's condition number (see
parity_util.conditioned_errors).
"""
import numpy as np
import pytest

from favor_inputs import (CAUSAL8K, DEMO64, LONG64K, MAP_ELU1, MAP_POSITIVE, MAP_RELU, MAP_TRIG,
                          MAP_TRIG_SOFTMAX, NC4096,
                          SWEEP16K, make_inputs, sweep_variants)
from parity_util import (causal_trig_condition, conditioned_errors, oracle_ref, row_errors,
                         run_gpu, scaled_inputs, to_device, trig_condition)

pytestmark = pytest.mark.gpu

F32_MAX = 1e-4
BF16_MAX = 2e-2
BF16_MEAN = 2e-3


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from favor_random_feature_gb300 import build
    build.build()


def check_bf16(e, what):
    assert e.max() <= BF16_MAX and e.mean() <= BF16_MEAN, \
        f"{what}: max {e.max():.3e} mean {e.mean():.3e}"


# ---------------------------------------------------------------------------
# fp32 entry point: the page's demo (B=H=1, L=64, d=32, m=256), 1e-4
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("fmap", [MAP_POSITIVE, MAP_TRIG, MAP_ELU1])
def test_demo64_fp32(causal, fmap):
    w = DEMO64.with_(feature_map=fmap, m=32 if fmap == MAP_ELU1 else 256)
    inp = make_inputs(w)
    out = run_gpu(inp, causal, fmap)
    ref = oracle_ref(inp, causal, fmap)
    e = row_errors(out, ref)
    assert e.max() <= F32_MAX, e.max()


@pytest.mark.parametrize("causal", [False, True])
def test_fp32_multihead_ragged(causal):
    w = NC4096.with_(dtype="f32")
    inp = make_inputs(w, L=333, B=2, H=3)
    e = row_errors(run_gpu(inp, causal, MAP_POSITIVE), oracle_ref(inp, causal, MAP_POSITIVE))
    assert e.max() <= F32_MAX, e.max()


# ---------------------------------------------------------------------------
# bf16 entry point, reduced sizes (several 128-token tiles + a ragged tail)
# ---------------------------------------------------------------------------
REDUCED = [
    (NC4096, False, 1000),
    (CAUSAL8K, True, 1000),
    (LONG64K, True, 1300),
    (LONG64K, False, 1300),
]


@pytest.mark.parametrize("w,causal,L", REDUCED, ids=lambda x: getattr(x, "name", str(x)))
def test_bf16_reduced(w, causal, L):
    inp = make_inputs(w, L=L, B=1, H=3)
    e = row_errors(run_gpu(inp, causal, MAP_POSITIVE), oracle_ref(inp, causal, MAP_POSITIVE))
    check_bf16(e, f"{w.name} L={L} causal={causal}")


@pytest.mark.parametrize("w", sweep_variants(), ids=lambda w: w.name)
def test_sweep_reduced(w):
    inp = make_inputs(w, L=700, B=1, H=2)
    fmap = w.feature_map
    out = run_gpu(inp, True, fmap)
    ref = oracle_ref(inp, True, fmap)
    if fmap == MAP_TRIG:
        e = conditioned_errors(out, ref, causal_trig_condition(inp), inp.v32)
    else:
        e = row_errors(out, ref)
    check_bf16(e, w.name)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d,m", [(64, 64), (64, 128), (128, 64), (128, 128), (128, 256), (128, 512)])
def test_trig_well_conditioned(causal, d, m):
    # q, k scaled by 1/4: |q-k|^2 ~ 1 (d = 64) or 1.4 (d = 128), so the
    # Gaussian kernel the sin/cos features estimate is O(1) and most
    # denominators are well conditioned; d = 128 is the sweep's head size,
    # scored here on the plain per-row metric
    w = SWEEP16K.with_(m=m, feature_map=MAP_TRIG, d=d, dv=d)
    inp = scaled_inputs(make_inputs(w, L=400, B=1, H=2), 0.25)
    out = run_gpu(inp, causal, MAP_TRIG)
    ref = oracle_ref(inp, causal, MAP_TRIG)
    kap = causal_trig_condition(inp) if causal else trig_condition(inp)
    good = kap <= 10
    assert good.mean() > 0.5
    e = row_errors(out[good][:, None, None, :], ref[good][:, None, None, :])
    check_bf16(e, "trig")


# ---------------------------------------------------------------------------
# edge cases
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("L", [1, 2, 127, 128, 129, 255, 257])
@pytest.mark.parametrize("causal", [False, True])
def test_short_and_ragged_lengths(L, causal):
    inp = make_inputs(CAUSAL8K, L=L, B=1, H=2)
    e = row_errors(run_gpu(inp, causal, MAP_POSITIVE), oracle_ref(inp, causal, MAP_POSITIVE))
    assert e.max() <= BF16_MAX, e.max()


@pytest.mark.parametrize("w,bar", [(SWEEP16K.with_(m=512), "bf16"), (NC4096.with_(dtype="f32"), "f32")],
                         ids=["d128-r512-bf16", "f32"])
def test_noncausal_chunk_ranges(w, bar):
    """The SIMT non-causal state is summed from up to 8 ranges of 64-row chunks:
    L = 1100 gives 18 chunks in ranges of 3, the last two ranges empty."""
    inp = make_inputs(w, L=1100, B=1, H=2)
    e = row_errors(run_gpu(inp, False, MAP_POSITIVE), oracle_ref(inp, False, MAP_POSITIVE))
    if bar == "f32":
        assert e.max() <= F32_MAX, e.max()
    else:
        check_bf16(e, w.name)


@pytest.mark.parametrize("d,dv,m", [(32, 32, 16), (32, 128, 64), (128, 32, 128), (64, 128, 256),
                                    (128, 64, 32)])
@pytest.mark.parametrize("causal", [False, True])
def test_head_dims(d, dv, m, causal):
    w = CAUSAL8K.with_(d=d, dv=dv, m=m, omega="iid")
    inp = make_inputs(w, L=300, B=2, H=1)
    e = row_errors(run_gpu(inp, causal, MAP_POSITIVE), oracle_ref(inp, causal, MAP_POSITIVE))
    check_bf16(e, f"d={d} dv={dv} m={m}")


# many heads: one segment per head (or two), so each CTA scans several chunks
# and carries its state from chunk to chunk (the launch shape of the full-size
# workloads, at a length the oracle finishes quickly)
@pytest.mark.parametrize("B,H,dv,heads", [(1, 160, 64, [0, 77, 159]), (4, 19, 64, [0, 40, 75]),
                                          (2, 20, 64, [0, 21, 39]), (2, 80, 128, [1, 100, 159])],
                         ids=["one_segment", "two_segments", "four_segments", "dv128"])
def test_causal_many_chunks_per_cta(B, H, dv, heads):
    w = CAUSAL8K.with_(dv=dv)
    inp = make_inputs(w, L=1000, B=B, H=H)
    out = run_gpu(inp, True, MAP_POSITIVE)
    ref = oracle_ref(inp, True, MAP_POSITIVE, heads=heads)
    BH = B * H
    e = row_errors(out.reshape(BH, 1000, dv)[heads], ref.reshape(BH, 1000, dv)[heads])
    check_bf16(e, f"B={B} H={H} dv={dv}")


@pytest.mark.parametrize("m,fmap", [(256, MAP_POSITIVE), (512, MAP_POSITIVE), (256, MAP_TRIG)],
                         ids=["pos-r256", "pos-r512", "trig-r512"])
def test_split_heads_many_segments(m, fmap):
    """One head of a split feature set (d = dv = 128): its clusters scan many
    segments, whose prefix states come from the state pass through the
    combine pass (one key reference for every feature slice)."""
    w = SWEEP16K.with_(m=m, feature_map=fmap)
    inp = make_inputs(w, L=3000, B=1, H=1)
    if fmap == MAP_TRIG:
        inp = scaled_inputs(inp, 0.25)
    out = run_gpu(inp, True, fmap)
    ref = oracle_ref(inp, True, fmap)
    if fmap == MAP_TRIG:
        kap = causal_trig_condition(inp)
        good = kap <= 10
        assert good.mean() > 0.5
        e = row_errors(out[good][:, None, None, :], ref[good][:, None, None, :])
    else:
        e = row_errors(out, ref)
    check_bf16(e, f"m={m} map={fmap}")


WIDENED = [(MAP_POSITIVE, 64, 64), (MAP_POSITIVE, 128, 64), (MAP_TRIG, 64, 32), (MAP_ELU1, 64, 64)]


@pytest.mark.parametrize("causal", [False, True], ids=["noncausal", "causal"])
@pytest.mark.parametrize("fmap,d,m", WIDENED, ids=["pos-d64", "pos-d128", "trig-d64", "elu1-d64"])
def test_r64_heads_on_the_tensor_cores(fmap, d, m, causal):
    """r = 64 features run on the tensor-core kernels as r = 128 with every
    projection taken twice (numerator and denominator double, the ratio does
    not change): the tensor-core kernels must run, and the rows must meet the
    bf16 bar against the oracle's r = 64 result."""
    import favor_random_feature_gb300 as fv
    w = SWEEP16K.with_(feature_map=fmap, d=d, dv=d, m=m, omega="iid")
    inp = make_inputs(w, L=700, B=1, H=2)
    if fmap == MAP_TRIG:
        inp = scaled_inputs(inp, 0.25)
    fv.favor_stats_enable(True)
    try:
        out = run_gpu(inp, causal, fmap)
        st = fv.favor_stats_read()
    finally:
        fv.favor_stats_enable(False)
    assert st.dominant_kernel.decode().startswith("tc_"), st.dominant_kernel
    ref = oracle_ref(inp, causal, fmap)
    if fmap == MAP_TRIG:
        kap = causal_trig_condition(inp) if causal else trig_condition(inp)
        good = kap <= 10
        assert good.mean() > 0.5
        e = row_errors(out[good][:, None, None, :], ref[good][:, None, None, :])
    else:
        e = row_errors(out, ref)
    check_bf16(e, f"r=64 map={fmap} d={d}")


@pytest.mark.parametrize("m,B", [(256, 2), (512, 1)], ids=["pairs", "quads"])
def test_split_heads_two_segments(m, B):
    """Two segments per head in the feature-split scan (d = dv = 128; the
    benchmark's launch shape for m = 256): the second segment's clusters sum
    the piece states of the first in their prologue (no combine pass)."""
    w = SWEEP16K.with_(m=m)
    inp = make_inputs(w, L=2048, B=B, H=8)
    BH = B * 8
    heads = [0, BH // 2 + 1, BH - 1]
    out = run_gpu(inp, True, MAP_POSITIVE)
    ref = oracle_ref(inp, True, MAP_POSITIVE, heads=heads)
    e = row_errors(out.reshape(BH, 2048, w.dv)[heads], ref.reshape(BH, 2048, w.dv)[heads])
    check_bf16(e, f"m={m} two segments")


def test_split_heads_many_pieces():
    """r = 1024 (eight-CTA clusters) on one head of 38 chunks: 19 segments
    whose states come in 36 pieces of 8 feature tiles, 288 (piece, tile)
    scales in the combine pass."""
    w = SWEEP16K.with_(m=1024, d=64, dv=64)
    inp = make_inputs(w, L=38 * 128, B=1, H=1)
    e = row_errors(run_gpu(inp, True, MAP_POSITIVE), oracle_ref(inp, True, MAP_POSITIVE))
    check_bf16(e, "m=1024 d=64 L=4864")


def test_causal_first_row_is_v0_and_last_row_matches_noncausal():
    inp = make_inputs(CAUSAL8K, L=300, B=1, H=2)
    oc = run_gpu(inp, True, MAP_POSITIVE)
    on = run_gpu(inp, False, MAP_POSITIVE)
    v0 = inp.v32[:, :, 0].astype(np.float64)
    assert np.max(np.abs(oc[:, :, 0] - v0)) <= 2e-2 * np.max(np.abs(v0))
    e = row_errors(oc[:, :, -1:], on[:, :, -1:])
    assert e.max() <= 1e-2


def test_deterministic():
    inp = make_inputs(CAUSAL8K, L=600, B=1, H=2)
    a = run_gpu(inp, True, MAP_POSITIVE)
    b = run_gpu(inp, True, MAP_POSITIVE)
    assert np.array_equal(a, b)


def test_constant_values():
    inp = make_inputs(CAUSAL8K, L=200, B=1, H=1)
    from favor_inputs import bf16_bits, bf16_to_f32
    vals = np.broadcast_to((np.arange(64, dtype=np.float32) - 20) / 8, inp.v32.shape).copy()
    inp.v = bf16_bits(vals)
    inp.v32 = bf16_to_f32(inp.v)
    for causal in (False, True):
        out = run_gpu(inp, causal, MAP_POSITIVE)
        assert np.allclose(out, inp.v32, rtol=5e-3, atol=5e-3)


@pytest.mark.parametrize("causal", [False, True], ids=["noncausal", "causal"])
@pytest.mark.parametrize("fmap,w", [(MAP_POSITIVE, CAUSAL8K), (MAP_ELU1, CAUSAL8K.with_(m=64)),
                                    (MAP_POSITIVE, NC4096.with_(dtype="f32"))],
                         ids=["positive", "elu1", "positive-f32"])
def test_zero_keys_give_the_mean_of_the_values(fmap, w, causal):
    """With every key zero, every key has the same features (1/sqrt(m) each for
    the positive map, all ones for ELU+1), so every query weighs the keys it
    sees equally whatever q and omega are: out_i is the mean of v over keys
    0..i (causal) or over all keys (non-causal).  A closed form, not the
    oracle; the tensor-core path (bf16) and the fp32 path."""
    from favor_inputs import bf16_bits
    inp = make_inputs(w.with_(feature_map=fmap), L=700, B=1, H=2)
    inp.k32 = np.zeros_like(inp.k32)
    inp.k = bf16_bits(inp.k32) if w.dtype == "bf16" else inp.k32
    out = run_gpu(inp, causal, fmap)
    v = inp.v32.astype(np.float64)
    if causal:
        want = np.cumsum(v, axis=2) / np.arange(1, v.shape[2] + 1)[:, None]
    else:
        want = np.broadcast_to(v.mean(axis=2, keepdims=True), v.shape)
    e = row_errors(out, want)
    if w.dtype == "bf16":
        check_bf16(e, f"zero keys map={fmap} causal={causal}")
    else:
        assert e.max() <= F32_MAX, e.max()


# ---------------------------------------------------------------------------
# the other entry points
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("fmap", [MAP_POSITIVE, MAP_TRIG, MAP_ELU1])
def test_feature_map_entry(fmap):
    import torch
    import favor_random_feature_gb300 as fv
    import oracle
    w = CAUSAL8K.with_(feature_map=fmap, m=64 if fmap == MAP_ELU1 else 128)
    inp = make_inputs(w, L=150, B=1, H=2)
    q, _, _, om = to_device(inp)
    r = fv.favor_feature_dim(fmap, w.d, w.m)
    phi = torch.empty((1, 2, 150, r), dtype=torch.float32, device="cuda")
    ls = torch.empty((1, 2, 150), dtype=torch.float32, device="cuda")
    rc = fv.favor_feature_map(q, om, phi, ls, 1, 2, 150, w.d, w.m, fmap, 0,
                              torch.cuda.current_stream())
    assert rc == 0
    got = phi.cpu().numpy().astype(np.float64) * np.exp(ls.cpu().numpy().astype(np.float64))[..., None]
    for h in range(2):
        want = oracle.features(inp.q32[0, h], None if fmap == MAP_ELU1 else inp.omega[h], fmap)
        # fp32 projections of size up to ~20 carry ~1e-6 absolute error into sin/cos
        assert np.allclose(got[0, h], want, rtol=1e-4, atol=3e-5 * np.abs(want).max())


@pytest.mark.parametrize("B,H,L,causal", [(1, 2, 500, True), (4, 3, 300, True), (6, 2, 257, False), (1, 1, 129, True),
                                          (2, 16, 300, True), (16, 4, 130, False)],
                         ids=["heads-split", "batch-groups", "uneven-batches", "one-head", "last-quarter",
                              "last-batch-and-quarter"])
def test_host_entry_matches_oracle(B, H, L, causal):
    """The host-buffer entry point copies in, computes and copies out head
    groups (whole batches, or head ranges of one batch) on overlapping streams;
    each group is its own forward pass, so its rows meet the same bar against
    the oracle as the device entry point's, and every row is written."""
    import favor_random_feature_gb300 as fv
    inp = make_inputs(CAUSAL8K, L=L, B=B, H=H)
    w = inp.w
    out = np.full((w.B, w.H, w.L, w.dv), np.nan, dtype=np.float32)
    om = np.ascontiguousarray(inp.omega, dtype=np.float32)
    rc = fv.favor_attn_forward_host(inp.q, inp.k, inp.v, om, out, w.B, w.H, w.L, w.d, w.dv,
                                    w.m, int(causal), MAP_POSITIVE)
    assert rc == 0, fv.strerror(rc)
    ref = oracle_ref(inp, causal, MAP_POSITIVE)
    check_bf16(row_errors(out.astype(np.float64), ref), "host entry")
    check_bf16(row_errors(run_gpu(inp, causal, MAP_POSITIVE), ref), "device entry")


@pytest.mark.parametrize("fmap", [MAP_TRIG, MAP_ELU1], ids=["trig", "elu1"])
def test_host_entry_other_maps(fmap):
    """The host-buffer entry point passes the feature map through to every
    head group: sin/cos (inputs scaled so the kernel is O(1), rows with
    condition <= 10 scored) and ELU+1 (no omega)."""
    import favor_random_feature_gb300 as fv
    inp = make_inputs(CAUSAL8K.with_(feature_map=fmap, m=64 if fmap == MAP_ELU1 else 128), L=400, B=2, H=8)
    if fmap == MAP_TRIG:
        inp = scaled_inputs(inp, 0.25)
    w = inp.w   # the shape of the arrays: the host entry point copies exactly that much
    out = np.full((w.B, w.H, w.L, w.dv), np.nan, dtype=np.float32)
    om = None if fmap == MAP_ELU1 else np.ascontiguousarray(inp.omega, dtype=np.float32)
    rc = fv.favor_attn_forward_host(inp.q, inp.k, inp.v, om, out, w.B, w.H, w.L, w.d, w.dv,
                                    w.m if fmap != MAP_ELU1 else w.d, 1, fmap)
    assert rc == 0, fv.strerror(rc)
    ref = oracle_ref(inp, True, fmap)
    got = out.astype(np.float64)
    if fmap == MAP_TRIG:
        good = causal_trig_condition(inp) <= 10
        assert good.mean() > 0.5
        e = row_errors(got[good][:, None, None, :], ref[good][:, None, None, :])
    else:
        e = row_errors(got, ref)
    check_bf16(e, f"host entry map={fmap}")


# ---------------------------------------------------------------------------
# full sizes, in the benchmark's launch configuration; oracle on sampled heads
# ---------------------------------------------------------------------------
FULL = [
    (NC4096, False, [0, 95]),
    (CAUSAL8K, True, [0, 37, 63]),
    (LONG64K, True, [0, 7]),
    (LONG64K, False, [3]),
]


@pytest.mark.parametrize("w,causal,heads", FULL, ids=lambda x: getattr(x, "name", str(x)))
def test_full_size_sampled_heads(w, causal, heads):
    inp = make_inputs(w)
    out = run_gpu(inp, causal, MAP_POSITIVE)
    ref = oracle_ref(inp, causal, MAP_POSITIVE, heads=heads)
    BH = w.B * w.H
    e = row_errors(out.reshape(BH, w.L, w.dv)[heads], ref.reshape(BH, w.L, w.dv)[heads])
    check_bf16(e, w.name)
    assert np.isfinite(out).all()


@pytest.mark.parametrize("m,heads", [(64, [5]), (128, [5]), (256, [5, 14]), (512, [5])])
def test_full_size_sweep_sampled(m, heads):
    """B=2, H=8, L=16384, d=dv=128 at full size in the launch configuration
    the benchmark times (m = 256: two-slice clusters, two segments; m = 512:
    four-slice clusters, one segment; m = 64, 128: whole heads)."""
    w = SWEEP16K.with_(m=m)
    inp = make_inputs(w)
    out = run_gpu(inp, True, MAP_POSITIVE)
    ref = oracle_ref(inp, True, MAP_POSITIVE, heads=heads)
    e = row_errors(out.reshape(16, w.L, w.dv)[heads], ref.reshape(16, w.L, w.dv)[heads])
    check_bf16(e, w.name)
    assert np.isfinite(out).all()


@pytest.mark.parametrize("fmap,m", [(MAP_ELU1, 128), (MAP_TRIG, 256)], ids=["elu1", "trig-m256"])
def test_full_size_sweep_other_maps(fmap, m):
    """Config 5's other maps at full size (B=2, H=8, L=16384, d=dv=128):
    ELU+1 (r = d = 128, whole heads) and sin/cos at m = 256 (r = 512,
    four-slice clusters), the latter on inputs scaled so the kernel is O(1)
    with the rows of condition <= 10 scored on the plain metric."""
    w = SWEEP16K.with_(feature_map=fmap, m=m)
    inp = make_inputs(w)
    if fmap == MAP_TRIG:
        inp = scaled_inputs(inp, 0.25)
    heads = [5]
    out = run_gpu(inp, True, fmap).reshape(16, w.L, w.dv)[heads]
    ref = oracle_ref(inp, True, fmap, heads=heads).reshape(16, w.L, w.dv)[heads]
    if fmap == MAP_TRIG:
        good = causal_trig_condition(inp, heads=heads).reshape(16, w.L)[heads] <= 10
        assert good.mean() > 0.5
        out, ref = out[good], ref[good]
    check_bf16(row_errors(out, ref), f"{w.name} map={fmap} full size")


@pytest.mark.parametrize("causal", [True, False], ids=["causal", "noncausal"])
def test_largest_accepted_shape(causal):
    """63 batch copies of the long64k heads (B = 63, H = 8, L = 65536, d = dv
    = 64, m = 256): q, k, v and out each hold 2.11e9 elements, just under the
    int32 element offsets the entry points accept (one batch more is refused
    on the host, tests/test_abi.py), and out spans 8.5 GB, so a 32-bit byte
    offset anywhere on the path would go wrong.  Every head is planned and
    computed the same way wherever it sits (one segment per head causal; the
    same pieces non-causal), so every batch copy must equal batch 0 bit for
    bit; batch 0 meets the bar against the oracle on sampled heads."""
    import torch
    import favor_random_feature_gb300 as fv
    inp = make_inputs(LONG64K)
    w = inp.w
    B = 63
    q0, k0, v0, om = to_device(inp)
    q = q0.expand(B, -1, -1, -1).contiguous()
    k = k0.expand(B, -1, -1, -1).contiguous()
    v = v0.expand(B, -1, -1, -1).contiguous()
    del q0, k0, v0
    assert 2 ** 31 - q.numel() <= 2 ** 25 and B * w.H * w.L * w.dv * 4 > 2 ** 32
    out = torch.empty((B, w.H, w.L, w.dv), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    try:
        rc = fv.favor_attn_forward(q, k, v, om, out, B, w.H, w.L, w.d, w.dv, w.m, int(causal), MAP_POSITIVE,
                                   stream)
        assert rc == fv.FAVOR_OK, fv.strerror(rc)
        st = fv.favor_get_device_status(stream)
        assert st == fv.FAVOR_OK, fv.strerror(st)
        same = [b for b in range(1, B) if torch.equal(out[b], out[0])]
        assert len(same) == B - 1, sorted(set(range(1, B)) - set(same))
        got = out[0].cpu().numpy().astype(np.float64)
    finally:
        del q, k, v, out
        torch.cuda.empty_cache()
    heads = [0, 7]
    ref = oracle_ref(inp, causal, MAP_POSITIVE, heads=heads)
    check_bf16(row_errors(got[heads], ref.reshape(w.H, w.L, w.dv)[heads]), "B=63 copies of long64k")



# ---------------------------------------------------------------------------
# the bf16 entry point runs the tensor-core kernels for the benchmark shapes
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("w,causal,kernel", [(CAUSAL8K, True, "tc_causal"),
                                             (NC4096, False, "tc_state"),
                                             (SWEEP16K.with_(m=128), True, "tc_causal"),
                                             (SWEEP16K.with_(m=64), True, "tc_causal")],
                         ids=["causal", "noncausal", "d128", "d128-r64"])
def test_tensor_core_path_taken(w, causal, kernel):
    import favor_random_feature_gb300 as fv
    inp = make_inputs(w, L=512, B=1, H=2)
    fv.favor_stats_enable(True)
    try:
        run_gpu(inp, causal, MAP_POSITIVE)
        st = fv.favor_stats_read()
    finally:
        fv.favor_stats_enable(False)
    assert st.dominant_kernel.decode() == kernel
    assert st.dominant_launches == 1 and st.kernel_launches >= 3


# ---------------------------------------------------------------------------
# many calls queued back to back on one stream, no host synchronisation in
# between: every bounded wait must still be met (a wait that runs out sets
# the device status) and the result must not change from call to call
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("w,causal", [(NC4096, False), (CAUSAL8K, True), (SWEEP16K, True)],
                         ids=["noncausal", "causal", "causal-split"])
def test_soak_status_stays_clean(w, causal):
    """Thousands of full-size calls queued without a host synchronisation:
    a wait whose barrier phase could be overtaken (a producer running ahead
    of its consumer) shows up as FAVOR_ERR_TIMEOUT in the status word."""
    import time
    import torch
    import favor_random_feature_gb300 as fv
    inp = make_inputs(w)
    q, k, v, om = to_device(inp)
    stream = torch.cuda.current_stream()
    out = torch.empty((w.B, w.H, w.L, w.dv), dtype=torch.float32, device="cuda")
    fv.favor_get_device_status(stream)
    t0, n = time.time(), 0
    while time.time() - t0 < 3.0:
        for _ in range(100):
            rc = fv.favor_attn_forward(q, k, v, om, out, w.B, w.H, w.L, w.d, w.dv, w.m, int(causal), MAP_POSITIVE,
                                       stream)
            assert rc == fv.FAVOR_OK, fv.strerror(rc)
        torch.cuda.synchronize()
        n += 100
    st = fv.favor_get_device_status(stream)
    assert st == fv.FAVOR_OK, (n, fv.strerror(st))


@pytest.mark.parametrize("w,causal", [(NC4096, False), (CAUSAL8K, True)], ids=["noncausal", "causal"])
def test_back_to_back_calls(w, causal):
    import torch
    import favor_random_feature_gb300 as fv
    inp = make_inputs(w)
    q, k, v, om = to_device(inp)
    stream = torch.cuda.current_stream()
    outs = [torch.empty((w.B, w.H, w.L, w.dv), dtype=torch.float32, device="cuda") for _ in range(2)]
    for i in range(24):
        rc = fv.favor_attn_forward(q, k, v, om, outs[i % 2], w.B, w.H, w.L, w.d, w.dv, w.m,
                                   int(causal), MAP_POSITIVE, stream)
        assert rc == fv.FAVOR_OK, fv.strerror(rc)
    torch.cuda.synchronize()
    st = fv.favor_get_device_status(stream)
    assert st == fv.FAVOR_OK, fv.strerror(st)
    assert torch.equal(outs[0], outs[1])


# ---------------------------------------------------------------------------
# ReLU and the softmax-scaled Fourier map (fp32 SIMT kernels for both entry
# points): fp32 arithmetic on the inputs' values, so the fp32 bar applies to
# both; the softmax-scaled map's denominators are not bounded away from zero,
# so its error is taken relative to each row's condition number
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("fmap", [MAP_RELU, MAP_TRIG_SOFTMAX], ids=["relu", "trig_softmax"])
def test_relu_and_softmax_scaled_trig(fmap, causal, dtype):
    w = NC4096.with_(feature_map=fmap, omega="iid", dtype=dtype, m=64 if fmap == MAP_RELU else 128)
    inp = make_inputs(w, L=333, B=2, H=3)
    out = run_gpu(inp, causal, fmap)
    ref = oracle_ref(inp, causal, fmap)
    if fmap == MAP_TRIG_SOFTMAX:
        cond = causal_trig_condition if causal else trig_condition
        e = conditioned_errors(out, ref, cond(inp, fmap=fmap), inp.v32)
    else:
        e = row_errors(out, ref)
    assert e.max() <= F32_MAX, e.max()


# ---------------------------------------------------------------------------
# bf16 output (favor_attn_forward_bf16out): the same computation as the fp32
# entry point with one final rounding, so the result is the fp32 output
# rounded to nearest even, bit for bit; against the oracle the bar grows by
# that rounding (2^-8 relative per row at most)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("w,causal,fmap,L", [
    (CAUSAL8K, True, MAP_POSITIVE, 1000),     # tensor-core scan
    (NC4096, False, MAP_POSITIVE, 1000),      # tensor-core state + output
    (CAUSAL8K, True, MAP_TRIG, 700),
    (NC4096.with_(omega="iid"), True, MAP_RELU, 333),   # SIMT kernels
    (NC4096.with_(omega="iid"), False, MAP_TRIG_SOFTMAX, 333),
    (SWEEP16K, True, MAP_POSITIVE, 700),     # feature-split scan (clusters of 2)
    (SWEEP16K.with_(m=512), True, MAP_POSITIVE, 700),   # clusters of 4, one receive slot
    (CAUSAL8K.with_(m=64), True, MAP_POSITIVE, 700),    # r = 64 widened to 128
    (NC4096.with_(m=64), False, MAP_POSITIVE, 700),
], ids=["causal", "noncausal", "trig_causal", "relu_simt", "trig_softmax_simt", "split2", "split4", "r64_causal",
        "r64_noncausal"])
def test_bf16_output(w, causal, fmap, L):
    import torch
    import favor_random_feature_gb300 as fv
    w = w.with_(feature_map=fmap, m=w.d if fmap == MAP_RELU else w.m)
    inp = make_inputs(w, L=L, B=1, H=3)
    q, k, v, om = to_device(inp)
    m = w.d if fmap == MAP_RELU else w.m
    out32 = torch.empty((1, 3, L, w.dv), dtype=torch.float32, device="cuda")
    out16 = torch.empty((1, 3, L, w.dv), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()
    assert fv.favor_attn_forward(q, k, v, om, out32, 1, 3, L, w.d, w.dv, m, int(causal), fmap, stream) == 0
    assert fv.favor_attn_forward_bf16out(q, k, v, om, out16, 1, 3, L, w.d, w.dv, m, int(causal), fmap,
                                         stream) == 0
    assert fv.favor_get_device_status(stream) == fv.FAVOR_OK
    assert torch.equal(out16, out32.to(torch.bfloat16))
    if fmap == MAP_POSITIVE:
        ref = oracle_ref(inp, causal, fmap)
        e = row_errors(out16.float().cpu().numpy().astype(np.float64), ref)
        assert e.max() <= BF16_MAX + 2 ** -8 and e.mean() <= BF16_MEAN + 2 ** -8, (e.max(), e.mean())
