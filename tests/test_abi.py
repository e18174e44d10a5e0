"""The C ABI library: it loads, exports every entry point include/favor.h
declares, and rejects bad arguments on the host before launching anything.
CPU only: no call here reaches a kernel."""
import os
import re

import pytest

import favor_random_feature_gb300 as fv
from favor_random_feature_gb300 import build as fbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    fbuild.build()
    return fv.lib()


def declared_symbols():
    txt = open(os.path.join(ROOT, "include", "favor.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(favor_\w+)\s*\(", txt)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert len(names) >= 8
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) <= set(fv.EXPORTS) | set(names)
    assert set(fv.EXPORTS) == set(names)


def test_strerror(lib):
    assert fv.strerror(0) == "FAVOR_OK"
    for s in (-1, -2, -3, -4, -5, -6):
        assert fv.strerror(s).startswith("FAVOR_ERR")
    assert "unknown" in fv.strerror(17)


def test_feature_dim(lib):
    assert fv.favor_feature_dim(fv.FAVOR_MAP_POSITIVE, 64, 256) == 256
    assert fv.favor_feature_dim(fv.FAVOR_MAP_TRIG, 64, 256) == 512
    assert fv.favor_feature_dim(fv.FAVOR_MAP_ELU1, 64, 64) == 64
    assert fv.favor_feature_dim(fv.FAVOR_MAP_ELU1, 64, 32) == -1
    assert fv.favor_feature_dim(7, 64, 64) == -1
    assert fv.favor_feature_dim(fv.FAVOR_MAP_RELU, 64, 64) == 64
    assert fv.favor_feature_dim(fv.FAVOR_MAP_RELU, 64, 128) == -1
    assert fv.favor_feature_dim(fv.FAVOR_MAP_TRIG_SOFTMAX, 64, 256) == 512
    assert fv.favor_feature_dim(5, 64, 64) == -1


# Fake, 16-byte aligned addresses: validation must reject these calls before
# touching them (or the GPU).
A, B_, C, W, O = 0x10000, 0x20000, 0x30000, 0x40000, 0x50000
GOOD = dict(B=1, H=2, L=64, d=64, dv=64, m=256, causal=0, feature_map=0)


def call(**kw):
    a = dict(q=A, k=B_, v=C, omega=W, out=O)
    a.update(GOOD)
    a.update(kw)
    return fv.favor_attn_forward(a["q"], a["k"], a["v"], a["omega"], a["out"], a["B"], a["H"],
                                 a["L"], a["d"], a["dv"], a["m"], a["causal"], a["feature_map"])


@pytest.mark.parametrize("kw,want", [
    (dict(q=None), fv.FAVOR_ERR_INVALID_ARG),
    (dict(k=None), fv.FAVOR_ERR_INVALID_ARG),
    (dict(v=None), fv.FAVOR_ERR_INVALID_ARG),
    (dict(out=None), fv.FAVOR_ERR_INVALID_ARG),
    (dict(omega=None), fv.FAVOR_ERR_INVALID_ARG),
    (dict(q=A + 2), fv.FAVOR_ERR_INVALID_ARG),          # misaligned
    (dict(out=A), fv.FAVOR_ERR_INVALID_ARG),            # aliases q
    (dict(B=0), fv.FAVOR_ERR_INVALID_ARG),
    (dict(H=-1), fv.FAVOR_ERR_INVALID_ARG),
    (dict(L=0), fv.FAVOR_ERR_INVALID_ARG),
    (dict(causal=2), fv.FAVOR_ERR_INVALID_ARG),
    (dict(feature_map=3), fv.FAVOR_ERR_INVALID_ARG),
    (dict(m=0), fv.FAVOR_ERR_INVALID_ARG),
    (dict(d=48), fv.FAVOR_ERR_UNSUPPORTED),
    (dict(dv=256), fv.FAVOR_ERR_UNSUPPORTED),
    (dict(m=100), fv.FAVOR_ERR_UNSUPPORTED),
    (dict(feature_map=2, m=32), fv.FAVOR_ERR_INVALID_ARG),   # elu1 needs m == d
    # a tensor of 2^31 elements or more: past the int32 element offsets
    (dict(B=64, H=8, L=65536), fv.FAVOR_ERR_UNSUPPORTED),            # 2^25 rows x d = 64
    (dict(B=32, H=8, L=65536, dv=128), fv.FAVOR_ERR_UNSUPPORTED),    # 2^24 rows x dv = 128
    (dict(B=1, H=1, L=2 ** 30, d=32, dv=32), fv.FAVOR_ERR_UNSUPPORTED),
])
def test_host_validation(lib, kw, want):
    assert call(**kw) == want


def test_f32_and_host_entry_validate_too(lib):
    assert fv.favor_attn_forward_f32(None, B_, C, W, O, 1, 1, 8, 32, 32, 16, 0, 0) == \
        fv.FAVOR_ERR_INVALID_ARG
    assert fv.favor_attn_forward_host(A, B_, C, None, O, 1, 1, 8, 32, 32, 16, 0, 0) == \
        fv.FAVOR_ERR_INVALID_ARG
    assert fv.favor_feature_map(A, W, O, None, 1, 1, 8, 32, 16, 0, 0) == fv.FAVOR_ERR_INVALID_ARG


def test_noalloc_rejects_scratch_beyond_its_maximum(lib):
    """The no-allocation entry point refuses a shape whose scratch exceeds its
    fixed array before any device work: B*H = 256 heads of L = 65536 need
    far more than 32 MiB of segment states.  The fake, far-apart pointers are
    never touched (on a machine without a GPU the same refusal holds)."""
    q, k, v, w, o = (i << 40 for i in range(1, 6))
    rc = fv.favor_attn_forward_noalloc(q, k, v, w, o, 16, 16, 65536, 64, 64, 256, 1, fv.FAVOR_MAP_POSITIVE)
    assert rc == fv.FAVOR_ERR_UNSUPPORTED
