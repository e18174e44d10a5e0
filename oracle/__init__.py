"""Float64 CPU oracle for the FAVOR+ forward pass -- test infrastructure only.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA
library (``favor_random_feature_gb300``) and never imports it.

The arithmetic lives in ``favor_oracle.c`` (plain C, float64, OpenMP over
heads).  This wrapper only compiles it (``build``) and marshals numpy arrays
to it.  Each function of the C file cites the passage of the pages it
follows.  Pins (tests/test_oracle.py) tie it to things other than itself:
the page's printed demo table, the closed-form kernel identity, brute-force
O(L^2) attention, Monte-Carlo unbiasedness with O(1/m) variance, the
softmax limit for large m, positivity, and invariances.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "favor_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")

MAP_POSITIVE, MAP_TRIG, MAP_ELU1, MAP_RELU, MAP_TRIG_SOFTMAX = 0, 1, 2, 3, 4
NO_OMEGA = (MAP_ELU1, MAP_RELU)   # elementwise maps: r = d, no projection

_lib = None


def build(force: bool = False) -> str:
    """Compile favor_oracle.c to oracle/_build/liboracle.so (gcc, float64,
    no FP contraction so results agree across host architectures)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    base = ["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fPIC", "-shared",
            _SRC, "-o", _LIB_PATH + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.POINTER(ctypes.c_double)
        lib.oracle_features.argtypes = [P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int, P]
        lib.oracle_features.restype = ctypes.c_int
        lib.oracle_forward.argtypes = [P, P, P, P, P, P] + [ctypes.c_int] * 8 + [
            ctypes.POINTER(ctypes.c_int), ctypes.c_int]
        lib.oracle_forward.restype = ctypes.c_int
        lib.oracle_feature_dim.argtypes = [ctypes.c_int] * 3
        lib.oracle_state.argtypes = [P] * 5 + [ctypes.c_int] * 7
        lib.oracle_state.restype = ctypes.c_int
        lib.oracle_decode_step.argtypes = [P] * 7 + [ctypes.c_int] * 6
        lib.oracle_decode_step.restype = ctypes.c_int
        U64 = ctypes.c_uint64
        lib.oracle_philox4x64.argtypes = [ctypes.POINTER(U64), ctypes.POINTER(U64), ctypes.POINTER(U64)]
        lib.oracle_philox4x64.restype = None
        lib.oracle_normal.argtypes = [U64, U64, U64]
        lib.oracle_normal.restype = ctypes.c_double
        lib.oracle_draw_omega.argtypes = [P] + [ctypes.c_int] * 4 + [U64]
        lib.oracle_draw_omega.restype = ctypes.c_int
        lib.oracle_backward.argtypes = [P] * 9 + [ctypes.c_int] * 8
        lib.oracle_backward.restype = ctypes.c_int
        lib.oracle_feature_dim.restype = ctypes.c_int
        _lib = lib
    return _lib


def _dp(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double)) if a is not None else None


def feature_dim(feature_map: int, d: int, m: int) -> int:
    return _load().oracle_feature_dim(feature_map, d, m)


def features(x, omega, feature_map: int = MAP_POSITIVE):
    """phi of the rows of x [n][d] with projection omega [m][d] -> [n][r] (float64)."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    n, d = x.shape
    if feature_map in NO_OMEGA:
        om, m = None, d
    else:
        om = np.ascontiguousarray(omega, dtype=np.float64)
        m = om.shape[0]
        assert om.shape[1] == d
    r = lib.oracle_feature_dim(feature_map, d, m)
    phi = np.empty((n, r), dtype=np.float64)
    rc = lib.oracle_features(_dp(x), _dp(om), n, d, m, feature_map, _dp(phi))
    if rc:
        raise FloatingPointError(f"oracle_features failed ({rc}): exponent out of range")
    return phi


def forward(q, k, v, omega, causal: bool, feature_map: int = MAP_POSITIVE,
            heads=None, return_den: bool = False):
    """FAVOR+ attention forward in float64.

    q, k: [B][H][L][d]; v: [B][H][L][dv]; omega: [H][m][d] (None for elu1).
    heads: optional iterable of flat head indices b*H+h; only those heads'
    rows are computed (the others are left NaN).  Returns out [B][H][L][dv]
    (and den [B][H][L] with return_den)."""
    lib = _load()
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    B, H, L, d = q.shape
    dv = v.shape[-1]
    assert k.shape == q.shape and v.shape[:3] == q.shape[:3]
    if feature_map in NO_OMEGA:
        om, m = None, d
    else:
        om = np.ascontiguousarray(omega, dtype=np.float64)
        assert om.shape[0] == H and om.shape[2] == d
        m = om.shape[1]
    out = np.full((B, H, L, dv), np.nan, dtype=np.float64)
    den = np.full((B, H, L), np.nan, dtype=np.float64) if return_den else None
    if heads is not None:
        hl = np.ascontiguousarray(np.asarray(list(heads), dtype=np.int32))
        hp, nh = hl.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), len(hl)
    else:
        hp, nh = None, 0
    rc = lib.oracle_forward(_dp(q), _dp(k), _dp(v), _dp(om), _dp(out), _dp(den),
                            B, H, L, d, dv, m, int(bool(causal)), feature_map, hp, nh)
    if rc:
        raise FloatingPointError(f"oracle_forward failed ({rc})")
    return (out, den) if return_den else out


def _omega_arg(omega, feature_map, H, d):
    if feature_map in NO_OMEGA:
        return None, d
    om = np.ascontiguousarray(omega, dtype=np.float64)
    assert om.shape[0] == H and om.shape[2] == d
    return om, om.shape[1]


def state(k, v, omega, feature_map: int = MAP_POSITIVE):
    """Carried state after all L keys of each head (float64):
    S [B][H][r][dv] = sum_j phi(k_j) v_j^T and z [B][H][r] = sum_j phi(k_j).
    k: [B][H][L][d]; v: [B][H][L][dv]; omega: [H][m][d] (None for elu1)."""
    lib = _load()
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    B, H, L, d = k.shape
    dv = v.shape[-1]
    assert v.shape[:3] == k.shape[:3]
    om, m = _omega_arg(omega, feature_map, H, d)
    r = lib.oracle_feature_dim(feature_map, d, m)
    S = np.empty((B, H, r, dv), dtype=np.float64)
    z = np.empty((B, H, r), dtype=np.float64)
    rc = lib.oracle_state(_dp(k), _dp(v), _dp(om), _dp(S), _dp(z), B, H, L, d, dv, m, feature_map)
    if rc:
        raise FloatingPointError(f"oracle_state failed ({rc})")
    return S, z


def decode_step(q, k, v, omega, S, z, feature_map: int = MAP_POSITIVE):
    """One decode step for every head: returns (out [B][H][dv], S', z') with
    S' = S + phi(k) v^T, z' = z + phi(k), out = phi(q)^T S' / phi(q)^T z'.
    q, k: [B][H][d]; v: [B][H][dv]; S, z as returned by ``state`` (not
    modified)."""
    lib = _load()
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    B, H, d = q.shape
    dv = v.shape[-1]
    assert k.shape == q.shape and v.shape[:2] == q.shape[:2]
    om, m = _omega_arg(omega, feature_map, H, d)
    S2 = np.array(S, dtype=np.float64, order="C", copy=True)
    z2 = np.array(z, dtype=np.float64, order="C", copy=True)
    r = lib.oracle_feature_dim(feature_map, d, m)
    assert S2.shape == (B, H, r, dv) and z2.shape == (B, H, r)
    out = np.empty((B, H, dv), dtype=np.float64)
    rc = lib.oracle_decode_step(_dp(q), _dp(k), _dp(v), _dp(om), _dp(S2), _dp(z2), _dp(out),
                                B, H, d, dv, m, feature_map)
    if rc:
        raise FloatingPointError(f"oracle_decode_step failed ({rc})")
    return out, S2, z2


def philox4x64(counter, key):
    """One Philox4x64-10 block: 4 counter words, 2 key words -> 4 uint64 words."""
    lib = _load()
    c = (ctypes.c_uint64 * 4)(*[int(x) for x in counter])
    k = (ctypes.c_uint64 * 2)(*[int(x) for x in key])
    o = (ctypes.c_uint64 * 4)()
    lib.oracle_philox4x64(c, k, o)
    return [int(x) for x in o]


def normal(seed: int, stream: int, e: int) -> float:
    """Normal number e of stream `stream` under `seed` (Philox4x64-10 + Box-Muller)."""
    return _load().oracle_normal(int(seed), int(stream), int(e))


def draw_omega(H: int, m: int, d: int, kind: int, seed: int):
    """omega [H][m][d] float64: kind 0 iid N(0, I) rows, 1 block-orthogonal."""
    lib = _load()
    out = np.empty((H, m, d), dtype=np.float64)
    rc = lib.oracle_draw_omega(_dp(out), H, m, d, kind, int(seed))
    if rc:
        raise ValueError(f"oracle_draw_omega failed ({rc})")
    return out


def backward(q, k, v, omega, g, causal: bool, feature_map: int = MAP_POSITIVE):
    """Gradients of a loss with dloss/dout = g through the forward pass:
    returns (dq, dk, dv, dw) float64; dw [H][m][d] is summed over the batch
    (None for the elementwise maps)."""
    lib = _load()
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    g = np.ascontiguousarray(g, dtype=np.float64)
    B, H, L, d = q.shape
    dv_ = v.shape[-1]
    assert k.shape == q.shape and v.shape[:3] == q.shape[:3] and g.shape == v.shape
    om, m = _omega_arg(omega, feature_map, H, d)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    dw = None if om is None else np.zeros((H, m, d), dtype=np.float64)
    rc = lib.oracle_backward(_dp(q), _dp(k), _dp(v), _dp(om), _dp(g), _dp(dq), _dp(dk), _dp(dv), _dp(dw),
                             B, H, L, d, dv_, m, int(bool(causal)), feature_map)
    if rc:
        raise FloatingPointError(f"oracle_backward failed ({rc})")
    return dq, dk, dv, dw


def threads_used() -> int:
    """OpenMP threads the oracle runs with (OMP_NUM_THREADS or all cores)."""
    env = os.environ.get("OMP_NUM_THREADS")
    return int(env) if env else (os.cpu_count() or 1)
