"""Helpers shared by the GPU parity tests: move seeded inputs to the device,
call the library through its C ABI, and measure the per-row normwise error
against the float64 oracle."""
import numpy as np

import favor_random_feature_gb300 as fv
from favor_inputs import MAP_ELU1, MAP_RELU, MAP_TRIG, MAP_TRIG_SOFTMAX

NO_OMEGA = (MAP_ELU1, MAP_RELU)


def to_device(inp):
    import torch
    w = inp.w
    if w.dtype == "bf16":
        conv = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(
            torch.bfloat16).cuda()
    else:
        conv = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()
    om = None
    if inp.omega is not None and w.feature_map not in NO_OMEGA:
        om = torch.from_numpy(np.ascontiguousarray(inp.omega, dtype=np.float32)).cuda()
    return conv(inp.q), conv(inp.k), conv(inp.v), om


def run_gpu(inp, causal, feature_map, entry=None):
    """Run the forward pass through the C ABI; returns out as float64 numpy."""
    import torch
    w = inp.w
    q, k, v, om = to_device(inp)
    out = torch.full((w.B, w.H, w.L, w.dv), float("nan"), dtype=torch.float32, device="cuda")
    m = w.d if feature_map in NO_OMEGA else w.m
    if entry is None:
        entry = fv.favor_attn_forward if w.dtype == "bf16" else fv.favor_attn_forward_f32
    stream = torch.cuda.current_stream()
    rc = entry(q, k, v, om, out, w.B, w.H, w.L, w.d, w.dv, m, int(causal), feature_map, stream)
    assert rc == fv.FAVOR_OK, fv.strerror(rc)
    st = fv.favor_get_device_status(stream)
    assert st == fv.FAVOR_OK, fv.strerror(st)
    return out.cpu().numpy().astype(np.float64)


def oracle_ref(inp, causal, feature_map, heads=None, return_den=False):
    import oracle
    om = None if feature_map in NO_OMEGA else inp.omega
    return oracle.forward(inp.q32, inp.k32, inp.v32, om, causal=causal,
                          feature_map=feature_map, heads=heads, return_den=return_den)


def row_errors(out, ref):
    """e_i = |o_i - ref_i|_2 / |ref_i|_2 per row (rows of ref that are NaN are skipped)."""
    out = out.reshape(-1, out.shape[-1])
    ref = ref.reshape(-1, ref.shape[-1])
    keep = ~np.isnan(ref).any(axis=1)
    out, ref = out[keep], ref[keep]
    assert np.isfinite(out).all(), "non-finite GPU output"
    return np.linalg.norm(out - ref, axis=1) / np.linalg.norm(ref, axis=1)


def trig_condition(inp, heads=None, fmap=MAP_TRIG):
    """kappa_i = (|phi(q_i)|^T sum_j |phi(k_j)|) / |phi(q_i)^T z| for the trig map
    (non-causal sums), used to select well-conditioned rows."""
    import oracle
    w = inp.w
    BH = w.B * w.H
    q = inp.q32.reshape(BH, w.L, w.d)
    k = inp.k32.reshape(BH, w.L, w.d)
    kap = np.full((BH, w.L), np.inf)
    for bh in (range(BH) if heads is None else heads):
        om = inp.omega[bh % w.H]
        pq = oracle.features(q[bh], om, fmap)
        pk = oracle.features(k[bh], om, fmap)
        kap[bh] = (np.abs(pq) @ np.abs(pk).sum(0)) / np.abs(pq @ pk.sum(0))
    return kap.reshape(w.B, w.H, w.L)


def causal_trig_condition(inp, heads=None, fmap=MAP_TRIG):
    import oracle
    w = inp.w
    BH = w.B * w.H
    q = inp.q32.reshape(BH, w.L, w.d)
    k = inp.k32.reshape(BH, w.L, w.d)
    kap = np.full((BH, w.L), np.inf)
    for bh in (range(BH) if heads is None else heads):
        om = inp.omega[bh % w.H]
        pq = oracle.features(q[bh], om, fmap)
        pk = oracle.features(k[bh], om, fmap)
        zabs = np.cumsum(np.abs(pk), axis=0)
        z = np.cumsum(pk, axis=0)
        kap[bh] = np.sum(np.abs(pq) * zabs, axis=1) / np.abs(np.sum(pq * z, axis=1))
    return kap.reshape(w.B, w.H, w.L)


def scaled_inputs(inp, s):
    """The same inputs with q and k multiplied by s (re-rounded to the storage type)."""
    import copy
    from favor_inputs import bf16_bits, bf16_to_f32
    out = copy.copy(inp)
    if inp.w.dtype == "bf16":
        out.q = bf16_bits(inp.q32 * np.float32(s))
        out.k = bf16_bits(inp.k32 * np.float32(s))
        out.q32, out.k32 = bf16_to_f32(out.q), bf16_to_f32(out.k)
    else:
        out.q = out.q32 = (inp.q32 * np.float32(s)).astype(np.float32)
        out.k = out.k32 = (inp.k32 * np.float32(s)).astype(np.float32)
    return out


def conditioned_errors(out, ref, kappa, v32):
    """Error of each row relative to its condition: |o_i - ref_i| /
    (kappa_i (max_j |v_j| + |ref_i|)).  For a result computed from features
    perturbed by a relative eps, this is at most about eps, however close the
    denominator comes to zero (used for the sin/cos map, whose denominators
    are not bounded away from zero)."""
    dv = out.shape[-1]
    o = out.reshape(-1, dv)
    r = ref.reshape(-1, dv)
    k = kappa.reshape(-1)
    vmax = np.linalg.norm(v32.reshape(-1, dv), axis=1).max()
    assert np.isfinite(o).all(), "non-finite GPU output"
    return np.linalg.norm(o - r, axis=1) / (k * (vmax + np.linalg.norm(r, axis=1)))
