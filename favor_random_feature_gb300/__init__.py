"""Thin Python binding of libfavor (include/favor.h): argument marshalling only.

Every step of the forward pass runs in the library's CUDA kernels; there is
no CPU or PyTorch fallback.  If libfavor.so has not been built, or a CUDA
device is missing, the calls raise.  PyTorch is used here only for device
memory and streams.

The entry points keep the C names and parameter order.  Tensor arguments may
be torch tensors (their data pointers are passed) or raw integer addresses.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libfavor.so")

FAVOR_OK = 0
FAVOR_ERR_INVALID_ARG = -1
FAVOR_ERR_UNSUPPORTED = -2
FAVOR_ERR_CUDA = -3
FAVOR_ERR_TIMEOUT = -4
FAVOR_ERR_NOMEM = -5
FAVOR_ERR_RANGE = -6

FAVOR_MAP_POSITIVE = 0
FAVOR_MAP_TRIG = 1
FAVOR_MAP_ELU1 = 2
FAVOR_MAP_RELU = 3
FAVOR_MAP_TRIG_SOFTMAX = 4

EXPORTS = (
    "favor_attn_forward",
    "favor_attn_forward_noalloc",
    "favor_attn_forward_bf16out",
    "favor_attn_forward_f32",
    "favor_attn_forward_host",
    "favor_feature_map",
    "favor_get_device_status",
    "favor_wait_expiry_check",
    "favor_strerror",
    "favor_release_workspace",
    "favor_feature_dim",
    "favor_stats_enable",
    "favor_stats_read",
    "favor_probe_ex2_rate",
    "favor_check_sincos",
    "favor_plan_info",
    "favor_state_floats",
    "favor_attn_state",
    "favor_attn_state_f32",
    "favor_attn_decode",
    "favor_attn_decode_f32",
    "favor_draw_omega",
    "favor_attn_backward",
    "favor_attn_backward_f32",
)

_lib = None


class FavorStats(ctypes.Structure):
    """favor_stats_t"""
    _fields_ = [("dominant_ms", ctypes.c_double), ("dominant_launches", ctypes.c_int),
                ("kernel_launches", ctypes.c_longlong), ("dominant_kernel", ctypes.c_char_p)]


class FavorError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {strerror(status)} ({status})")


def lib() -> ctypes.CDLL:
    """Load libfavor.so (built by ``build.build()``); raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libfavor.so is not built ({LIB_PATH}); run "
                               "favor_random_feature_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        vp, i, fp = ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p
        fwd = [vp, vp, vp, fp, fp] + [i] * 8 + [vp]
        for name in ("favor_attn_forward", "favor_attn_forward_f32", "favor_attn_forward_host",
                     "favor_attn_forward_noalloc", "favor_attn_forward_bf16out"):
            getattr(L, name).argtypes = fwd
            getattr(L, name).restype = i
        L.favor_feature_map.argtypes = [vp, fp, fp, fp] + [i] * 7 + [vp]
        L.favor_feature_map.restype = i
        L.favor_get_device_status.argtypes = [vp]
        L.favor_get_device_status.restype = i
        L.favor_wait_expiry_check.argtypes = [ctypes.c_longlong, vp]
        L.favor_wait_expiry_check.restype = i
        L.favor_strerror.argtypes = [i]
        L.favor_strerror.restype = ctypes.c_char_p
        L.favor_release_workspace.argtypes = []
        L.favor_release_workspace.restype = None
        L.favor_feature_dim.argtypes = [i, i, i]
        L.favor_feature_dim.restype = i
        L.favor_stats_enable.argtypes = [i]
        L.favor_stats_enable.restype = i
        L.favor_stats_read.argtypes = [ctypes.POINTER(FavorStats)]
        L.favor_stats_read.restype = i
        L.favor_probe_ex2_rate.argtypes = [ctypes.POINTER(ctypes.c_double), vp]
        L.favor_probe_ex2_rate.restype = i
        L.favor_check_sincos.argtypes = [vp, vp, vp, i, vp]
        L.favor_check_sincos.restype = i
        L.favor_plan_info.argtypes = [i] * 9 + [vp]
        L.favor_plan_info.restype = i
        L.favor_state_floats.argtypes = [i, i, i, i]
        L.favor_state_floats.restype = i
        for name in ("favor_attn_state", "favor_attn_state_f32"):
            getattr(L, name).argtypes = [vp, vp, fp, fp] + [i] * 7 + [vp]
            getattr(L, name).restype = i
        for name in ("favor_attn_backward", "favor_attn_backward_f32"):
            getattr(L, name).argtypes = [vp, vp, vp, fp, fp, fp, fp, fp, fp] + [i] * 8 + [vp]
            getattr(L, name).restype = i
        L.favor_draw_omega.argtypes = [fp, i, i, i, i, ctypes.c_ulonglong, vp]
        L.favor_draw_omega.restype = i
        for name in ("favor_attn_decode", "favor_attn_decode_f32"):
            getattr(L, name).argtypes = [vp, vp, vp, fp, fp, fp] + [i] * 6 + [vp]
            getattr(L, name).restype = i
        _lib = L
    return _lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):          # numpy array (host entry point)
        return x.ctypes.data
    raise TypeError(f"cannot pass {type(x)} as a pointer")


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream               # torch.cuda.Stream


def strerror(status: int) -> str:
    return lib().favor_strerror(int(status)).decode()


def favor_attn_forward(q, k, v, omega, out, B, H, L, d, dv, m, causal, feature_map, stream=None):
    return lib().favor_attn_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(omega), _ptr(out),
                                    B, H, L, d, dv, m, int(causal), int(feature_map),
                                    _stream(stream))


def favor_attn_forward_noalloc(q, k, v, omega, out, B, H, L, d, dv, m, causal, feature_map,
                               stream=None):
    return lib().favor_attn_forward_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(omega), _ptr(out),
                                            B, H, L, d, dv, m, int(causal), int(feature_map),
                                            _stream(stream))


def favor_attn_forward_bf16out(q, k, v, omega, out, B, H, L, d, dv, m, causal, feature_map, stream=None):
    return lib().favor_attn_forward_bf16out(_ptr(q), _ptr(k), _ptr(v), _ptr(omega), _ptr(out),
                                            B, H, L, d, dv, m, int(causal), int(feature_map),
                                            _stream(stream))


def favor_attn_forward_f32(q, k, v, omega, out, B, H, L, d, dv, m, causal, feature_map,
                           stream=None):
    return lib().favor_attn_forward_f32(_ptr(q), _ptr(k), _ptr(v), _ptr(omega), _ptr(out),
                                        B, H, L, d, dv, m, int(causal), int(feature_map),
                                        _stream(stream))


def favor_attn_forward_host(q, k, v, omega, out, B, H, L, d, dv, m, causal, feature_map,
                            stream=None):
    return lib().favor_attn_forward_host(_ptr(q), _ptr(k), _ptr(v), _ptr(omega), _ptr(out),
                                         B, H, L, d, dv, m, int(causal), int(feature_map),
                                         _stream(stream))


def favor_feature_map(x, omega, phi, log_scale, B, H, L, d, m, feature_map, is_key,
                      stream=None):
    return lib().favor_feature_map(_ptr(x), _ptr(omega), _ptr(phi), _ptr(log_scale),
                                   B, H, L, d, m, int(feature_map), int(is_key), _stream(stream))


def favor_get_device_status(stream=None) -> int:
    return lib().favor_get_device_status(_stream(stream))


def favor_wait_expiry_check(limit_cycles: int, stream=None) -> int:
    return lib().favor_wait_expiry_check(int(limit_cycles), _stream(stream))


def favor_release_workspace() -> None:
    lib().favor_release_workspace()


def favor_feature_dim(feature_map: int, d: int, m: int) -> int:
    return lib().favor_feature_dim(int(feature_map), int(d), int(m))


def favor_stats_enable(enable: bool) -> int:
    return lib().favor_stats_enable(int(bool(enable)))


def favor_stats_read() -> FavorStats:
    st = FavorStats()
    rc = lib().favor_stats_read(ctypes.byref(st))
    if rc != FAVOR_OK:
        raise FavorError(rc, "favor_stats_read")
    return st


def favor_plan_info(B, H, L, d, dv, m, causal, feature_map, sms):
    """(status, plan): the tensor-core launch plan of a shape on `sms` SMs
    (seven integers, the order include/favor.h gives)."""
    plan = (ctypes.c_int * 7)()
    rc = lib().favor_plan_info(int(B), int(H), int(L), int(d), int(dv), int(m), int(causal), int(feature_map),
                               int(sms), ctypes.cast(plan, ctypes.c_void_p))
    return rc, list(plan)


def favor_check_sincos(x, s, c, n, stream=None) -> int:
    return lib().favor_check_sincos(_ptr(x), _ptr(s), _ptr(c), int(n), _stream(stream))


def favor_probe_ex2_rate(stream=None) -> float:
    """Exponentials per second of the current device (favor.h)."""
    rate = ctypes.c_double(0.0)
    rc = lib().favor_probe_ex2_rate(ctypes.byref(rate), _stream(stream))
    if rc != FAVOR_OK:
        raise FavorError(rc, "favor_probe_ex2_rate")
    return rate.value


def favor_state_floats(d, dv, m, feature_map) -> int:
    return lib().favor_state_floats(int(d), int(dv), int(m), int(feature_map))


def favor_attn_state(k, v, omega, state, B, H, L, d, dv, m, feature_map, stream=None):
    return lib().favor_attn_state(_ptr(k), _ptr(v), _ptr(omega), _ptr(state), B, H, L, d, dv, m,
                                  int(feature_map), _stream(stream))


def favor_attn_state_f32(k, v, omega, state, B, H, L, d, dv, m, feature_map, stream=None):
    return lib().favor_attn_state_f32(_ptr(k), _ptr(v), _ptr(omega), _ptr(state), B, H, L, d, dv, m,
                                      int(feature_map), _stream(stream))


def favor_attn_decode(q, k, v, omega, state, out, B, H, d, dv, m, feature_map, stream=None):
    return lib().favor_attn_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(omega), _ptr(state), _ptr(out),
                                   B, H, d, dv, m, int(feature_map), _stream(stream))


def favor_attn_decode_f32(q, k, v, omega, state, out, B, H, d, dv, m, feature_map, stream=None):
    return lib().favor_attn_decode_f32(_ptr(q), _ptr(k), _ptr(v), _ptr(omega), _ptr(state), _ptr(out),
                                       B, H, d, dv, m, int(feature_map), _stream(stream))


def favor_attn_backward(q, k, v, omega, dout, dq, dk, dv, domega, B, H, L, d, dv_, m, causal, feature_map,
                        stream=None):
    return lib().favor_attn_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(omega), _ptr(dout), _ptr(dq), _ptr(dk),
                                     _ptr(dv), _ptr(domega), B, H, L, d, dv_, m, int(causal), int(feature_map),
                                     _stream(stream))


def favor_attn_backward_f32(q, k, v, omega, dout, dq, dk, dv, domega, B, H, L, d, dv_, m, causal, feature_map,
                            stream=None):
    return lib().favor_attn_backward_f32(_ptr(q), _ptr(k), _ptr(v), _ptr(omega), _ptr(dout), _ptr(dq), _ptr(dk),
                                         _ptr(dv), _ptr(domega), B, H, L, d, dv_, m, int(causal),
                                         int(feature_map), _stream(stream))


def favor_draw_omega(omega, H, m, d, kind, seed, stream=None):
    return lib().favor_draw_omega(_ptr(omega), int(H), int(m), int(d), int(kind), int(seed),
                                  _stream(stream))


def attention(q, k, v, omega, causal: bool, feature_map: int = FAVOR_MAP_POSITIVE,
              out=None, stream=None):
    """Convenience wrapper on torch CUDA tensors: q, k [B,H,L,d] and v
    [B,H,L,dv] (bfloat16 or float32, the same dtype), omega [H,m,d] float32
    (None for elu1 and relu).  Returns out [B,H,L,dv] float32."""
    import torch
    B, H, L, d = q.shape
    dv = v.shape[-1]
    m = d if feature_map in (FAVOR_MAP_ELU1, FAVOR_MAP_RELU) else omega.shape[1]
    if out is None:
        out = torch.empty((B, H, L, dv), dtype=torch.float32, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    fn = favor_attn_forward if q.dtype == torch.bfloat16 else favor_attn_forward_f32
    rc = fn(q, k, v, omega, out, B, H, L, d, dv, m, causal, feature_map, stream)
    if rc != FAVOR_OK:
        raise FavorError(rc, fn.__name__)
    return out
