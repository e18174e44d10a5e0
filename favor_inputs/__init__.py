"""Seeded synthetic inputs for the FAVOR+ forward pass.

This module only draws random numbers and rounds them to the storage
precision; it holds none of the method's arithmetic.  Both the CUDA path
(through the tests and the benchmark) and the float64 oracle read the values
made here, so that both sides see bit-identical inputs and the same random
projection omega.

Workloads (the pages' own demo plus the synthetic shapes of the Performer
setting "r=256 at d=64" of the Performer study notes, "Pitfalls"):

  demo64   B=H=1, L=64, d=dv=32, m=256, fp32.  Q, K, V drawn exactly as in the
           Linear Attention / Performer page, In[26] (legacy MT19937 seed 42,
           Q,K scaled by 0.3); omega from seed 0 as in its In[25], without the
           snippet's 1/sqrt(d) factor (the FAVOR+ equation of that page draws
           omega_i ~ N(0, I)).
  nc4096   B=8,  H=12, L=4096,  d=dv=64,  m=256, bf16, non-causal, block-orthogonal
  causal8k B=4,  H=16, L=8192,  d=dv=64,  m=256, bf16, causal, block-orthogonal
  long64k  B=1,  H=8,  L=65536, d=dv=64,  m=256, bf16, causal and non-causal, iid
  sweep16k B=2,  H=8,  L=16384, d=dv=128, m in {64,128,256,512}, bf16, causal,
           feature maps positive / trig / elu1, iid

q, k ~ N(0,1) * d^-1/4 and v ~ N(0,1) for the bf16 workloads: folding the
1/sqrt(d) softmax temperature into q and k, because the softmax kernel of the
pages is exp(q^T k) without the scale (Kernel Feature Maps page, "softmax
kernel").  Draw order: q, k, v, then omega head by head.
"""
from __future__ import annotations

import dataclasses

import numpy as np

# feature-map codes shared by every layer (same values as favor.h)
MAP_POSITIVE = 0
MAP_TRIG = 1
MAP_ELU1 = 2
MAP_RELU = 3
MAP_TRIG_SOFTMAX = 4
MAP_NAMES = {MAP_POSITIVE: "positive", MAP_TRIG: "trig", MAP_ELU1: "elu1", MAP_RELU: "relu",
             MAP_TRIG_SOFTMAX: "trig_softmax"}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    L: int
    d: int
    dv: int
    m: int
    causal: bool
    feature_map: int
    dtype: str          # "f32" or "bf16" storage of q, k, v
    omega: str          # "iid", "block_orth" or "page" (demo draw)
    seed: int

    @property
    def r(self) -> int:
        """Feature dimension: m (positive), 2m (trig, softmax-scaled trig), d (elu+1, relu)."""
        if self.feature_map in (MAP_TRIG, MAP_TRIG_SOFTMAX):
            return 2 * self.m
        if self.feature_map in (MAP_ELU1, MAP_RELU):
            return self.d
        return self.m

    @property
    def tokens(self) -> int:
        return self.B * self.H * self.L

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


DEMO64 = Workload("demo64", 1, 1, 64, 32, 32, 256, False, MAP_POSITIVE, "f32", "page", 42)
NC4096 = Workload("nc4096", 8, 12, 4096, 64, 64, 256, False, MAP_POSITIVE, "bf16", "block_orth", 1)
CAUSAL8K = Workload("causal8k", 4, 16, 8192, 64, 64, 256, True, MAP_POSITIVE, "bf16", "block_orth", 2)
LONG64K = Workload("long64k", 1, 8, 65536, 64, 64, 256, True, MAP_POSITIVE, "bf16", "iid", 3)
SWEEP16K = Workload("sweep16k", 2, 8, 16384, 128, 128, 256, True, MAP_POSITIVE, "bf16", "iid", 4)

WORKLOADS = {w.name: w for w in (DEMO64, NC4096, CAUSAL8K, LONG64K, SWEEP16K)}


def sweep_variants():
    """The feature-map / width sweep: positive and trig at m in {64..512}, elu1 at m=d."""
    out = []
    for m in (64, 128, 256, 512):
        out.append(SWEEP16K.with_(m=m, feature_map=MAP_POSITIVE, name=f"sweep16k_pos_m{m}"))
        out.append(SWEEP16K.with_(m=m, feature_map=MAP_TRIG, name=f"sweep16k_trig_m{m}"))
    out.append(SWEEP16K.with_(m=SWEEP16K.d, feature_map=MAP_ELU1, name="sweep16k_elu1"))
    return out


# ----------------------------------------------------------------------------
# bf16 storage: round-to-nearest-even of the fp32 value, as raw uint16 bits
# ----------------------------------------------------------------------------
def bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit pattern (uint16), round to nearest, ties to even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + rounding) >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit pattern (uint16) -> exact fp32 value."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# ----------------------------------------------------------------------------
# omega: the random projection, [H][m][d] fp32 (an input, not drawn inside)
# ----------------------------------------------------------------------------
def omega_iid(rng: np.random.Generator, H: int, m: int, d: int) -> np.ndarray:
    """omega_i ~ N(0, I_d), independent per head (FAVOR+ equation, both pages)."""
    return rng.standard_normal((H, m, d)).astype(np.float32)


def omega_block_orthogonal(rng: np.random.Generator, H: int, m: int, d: int) -> np.ndarray:
    """Block-orthogonal omega: per head, ceil(m/d) independent d x d Gaussian
    blocks whose rows are made orthonormal by modified Gram-Schmidt, each row
    then given an independent chi(d) length |g|, g ~ N(0, I_d), so that every
    row is still marginally N(0, I_d).  The last block keeps its first
    m - (nb-1) d rows.  (The 'O' of FAVOR+: orthogonal random features.)"""
    nb = -(-m // d)
    out = np.empty((H, m, d), dtype=np.float64)
    for h in range(H):
        rows = []
        for _ in range(nb):
            g = rng.standard_normal((d, d))
            q = np.empty_like(g)
            for i in range(d):
                v = g[i].copy()
                for j in range(i):
                    v -= np.dot(q[j], v) * q[j]
                q[i] = v / np.linalg.norm(v)
            lengths = np.sqrt(np.sum(rng.standard_normal((d, d)) ** 2, axis=1))
            rows.append(q * lengths[:, None])
        out[h] = np.concatenate(rows, axis=0)[:m]
    return out.astype(np.float32)


def omega_page(m: int, d: int) -> np.ndarray:
    """The pages' demo projection: legacy seed 0, randn(d, m), transposed to
    [1][m][d], WITHOUT the snippet's extra 1/sqrt(d) (see module docstring)."""
    rs = np.random.RandomState(0)
    w = rs.randn(d, m)
    return np.ascontiguousarray(w.T[None]).astype(np.float32)


# ----------------------------------------------------------------------------
# inputs
# ----------------------------------------------------------------------------
@dataclasses.dataclass
class Inputs:
    """q, k, v as stored for the GPU (fp32 array or bf16 bits), their exact
    values as float32 (for the oracle, which widens them to float64), and
    omega [H][m][d] fp32 (None for elu1)."""
    w: Workload
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    omega: np.ndarray | None
    q32: np.ndarray
    k32: np.ndarray
    v32: np.ndarray


def _store(x32: np.ndarray, dtype: str):
    if dtype == "bf16":
        bits = bf16_bits(x32)
        return bits, bf16_to_f32(bits)
    x32 = np.ascontiguousarray(x32, dtype=np.float32)
    return x32, x32


def make_inputs(w: Workload, L: int | None = None, B: int | None = None, H: int | None = None) -> Inputs:
    """Draw the workload's inputs.  L/B/H override the shape (same recipe,
    same seed) for reduced-size parity cases."""
    L = w.L if L is None else L
    B = w.B if B is None else B
    H = w.H if H is None else H
    if w.omega == "page":
        rs = np.random.RandomState(w.seed)
        q = (rs.randn(L, w.d).astype(np.float32) * 0.3).reshape(1, 1, L, w.d)
        k = (rs.randn(L, w.d).astype(np.float32) * 0.3).reshape(1, 1, L, w.d)
        v = rs.randn(L, w.dv).astype(np.float32).reshape(1, 1, L, w.dv)
        if B != 1 or H != 1:
            raise ValueError("the page's demo draw is a single head")
        om = omega_page(w.m, w.d) if w.feature_map not in (MAP_ELU1, MAP_RELU) else None
    else:
        rng = np.random.default_rng(w.seed)
        s = w.d ** -0.25
        q = rng.standard_normal((B, H, L, w.d), dtype=np.float32) * np.float32(s)
        k = rng.standard_normal((B, H, L, w.d), dtype=np.float32) * np.float32(s)
        v = rng.standard_normal((B, H, L, w.dv), dtype=np.float32)
        if w.feature_map in (MAP_ELU1, MAP_RELU):
            om = None
        elif w.omega == "block_orth":
            om = omega_block_orthogonal(rng, H, w.m, w.d)
        else:
            om = omega_iid(rng, H, w.m, w.d)
    qs, q32 = _store(q, w.dtype)
    ks, k32 = _store(k, w.dtype)
    vs, v32 = _store(v, w.dtype)
    return Inputs(w.with_(L=L, B=B, H=H), qs, ks, vs, om, q32, k32, v32)

