"""Thin ctypes binding of ``libh2o_gb300.so`` with the C ABI's names.

Argument marshalling only: every device-memory argument is a raw pointer
(an ``int``) or any object with ``data_ptr()`` (a torch tensor), every host
buffer of the state calls is a numpy array, and streams are ``cudaStream_t``
values (``int``) or objects with a ``cuda_stream`` attribute.  All compute
runs in the library; a failing call raises ``H2OError`` with the library's
message.  Importing this module does not load the library; the first call
does, and raises if the library was not built (there is no fallback).
"""
import ctypes
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libh2o_gb300.so")

H2O_OK = 0
H2O_ERR_ARG = -1
H2O_ERR_STATE = -2
H2O_ERR_ALLOC = -3
H2O_ERR_CUDA = -4
H2O_ERR_DEVICE_TIMEOUT = -5
H2O_ERR_UNSUPPORTED = -6
H2O_F32 = 0
H2O_BF16 = 1
H2O_KV8 = 2

# every symbol include/h2o.h declares, with (restype, argtypes)
_vp = ctypes.c_void_p
_i = ctypes.c_int
_d = ctypes.c_double
SIGNATURES = {
    "h2o_init": (_i, [ctypes.POINTER(_vp), _i, _i, _i, _i, _i, _i, _i, _d, _vp]),
    "h2o_init_gqa": (_i, [ctypes.POINTER(_vp), _i, _i, _i, _i, _i, _i, _i, _i, _d, _vp]),
    "sh_init": (_i, [ctypes.POINTER(_vp), _i, _i, _i, _i, _i, _i, _i, _d, _vp]),
    "sh_prefill": (_i, [_vp, _vp, _vp, _vp, _i]),
    "sh_decode_step": (_i, [_vp, _vp, _vp, _vp, _vp, _vp]),
    "h2o_prefill": (_i, [_vp, _vp, _vp, _vp, _i]),
    "h2o_decode_step": (_i, [_vp, _vp, _vp, _vp, _vp, _vp]),
    "lsh_init": (_i, [ctypes.POINTER(_vp), _i, _i, _i, _i, _i, _i, _d, _vp, _vp]),
    "lsh_prefill": (_i, [_vp, _vp, _vp, _vp, _i]),
    "lsh_decode_step": (_i, [_vp, _vp, _vp, _vp, _vp, _vp]),
    "h2o_get_state": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "h2o_set_state": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "h2o_get_prefill_stats": (_i, [_vp, _vp, _vp, _vp]),
    "h2o_get_kv_scales": (_i, [_vp, _vp, _vp]),
    "h2o_set_kv_scales": (_i, [_vp, _vp, _vp]),
    "h2o_set_stream": (_i, [_vp, _vp]),
    "h2o_set_decode_split": (_i, [_vp, _i]),
    "h2o_sync": (_i, [_vp]),
    "h2o_destroy": (None, [_vp]),
    "h2o_last_error": (ctypes.c_char_p, []),
    "h2o_prompt_scores_noalloc": (_i, [_vp, _vp, _i, _i, _i, _i, _i, _d, _vp, _vp]),
    "h2o_selftest_wait_timeout": (_i, [_vp]),
}

H2O_NOALLOC_MAX_TOKENS = 1 << 20

_lib = None


class H2OError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__("h2o status %d: %s" % (code, msg))
        self.code = code


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libh2o_gb300.so is not built (%s); run __graft_entry__.build()" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if isinstance(x, np.ndarray):
        if not x.flags["C_CONTIGUOUS"]:
            raise ValueError("host array must be C-contiguous")
        return x.ctypes.data
    if hasattr(x, "data_ptr"):
        if hasattr(x, "is_contiguous") and not x.is_contiguous():
            raise ValueError("tensor must be contiguous")
        return x.data_ptr()
    raise TypeError("cannot take a pointer of %r" % type(x))


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(rc):
    if rc != H2O_OK:
        raise H2OError(rc, h2o_last_error())


def h2o_last_error():
    return lib().h2o_last_error().decode()


def h2o_init(budget, heavy, recent, batch, heads, head_dim, dtype, scale, stream=None):
    h = _vp()
    _check(lib().h2o_init(ctypes.byref(h), budget, heavy, recent, batch, heads, head_dim, dtype,
                          float(scale), _stream(stream)))
    return h.value


def h2o_init_gqa(budget, heavy, recent, batch, kv_heads, groups, head_dim, dtype, scale, stream=None):
    h = _vp()
    _check(lib().h2o_init_gqa(ctypes.byref(h), budget, heavy, recent, batch, kv_heads, groups, head_dim,
                              dtype, float(scale), _stream(stream)))
    return h.value


def lsh_init(budget, recent, batch, heads, head_dim, dtype, scale, W, stream=None):
    h = _vp()
    _check(lib().lsh_init(ctypes.byref(h), budget, recent, batch, heads, head_dim, dtype, float(scale),
                          _ptr(W), _stream(stream)))
    return h.value


def h2o_prefill(h, Q, K, V, T):
    _check(lib().h2o_prefill(h, _ptr(Q), _ptr(K), _ptr(V), int(T)))


def lsh_prefill(h, Q, K, V, T):
    _check(lib().lsh_prefill(h, _ptr(Q), _ptr(K), _ptr(V), int(T)))


def h2o_decode_step(h, q, k, v, out, victim_out=None):
    _check(lib().h2o_decode_step(h, _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(victim_out)))


def lsh_decode_step(h, q, k, v, out, victim_out=None):
    _check(lib().lsh_decode_step(h, _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(victim_out)))


def sh_init(budget, heavy, recent, batch, heads, head_dim, dtype, scale, stream=None):
    h = _vp()
    _check(lib().sh_init(ctypes.byref(h), budget, heavy, recent, batch, heads, head_dim, dtype,
                         float(scale), _stream(stream)))
    return h.value


def sh_prefill(h, Q, K, V, T):
    _check(lib().sh_prefill(h, _ptr(Q), _ptr(K), _ptr(V), int(T)))


def sh_decode_step(h, q, k, v, out, victim_out=None):
    _check(lib().sh_decode_step(h, _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(victim_out)))


def h2o_get_state(h, K=None, V=None, score=None, pos=None, code=None, occupancy=None, next_pos=None):
    _check(lib().h2o_get_state(h, _ptr(K), _ptr(V), _ptr(score), _ptr(pos), _ptr(code), _ptr(occupancy),
                               _ptr(next_pos)))


def h2o_set_state(h, K=None, V=None, score=None, pos=None, code=None, occupancy=None, next_pos=None):
    _check(lib().h2o_set_state(h, _ptr(K), _ptr(V), _ptr(score), _ptr(pos), _ptr(code), _ptr(occupancy),
                               _ptr(next_pos)))


def h2o_get_prefill_stats(h, m=None, l=None, c=None):
    _check(lib().h2o_get_prefill_stats(h, _ptr(m), _ptr(l), _ptr(c)))


def h2o_get_kv_scales(h, kscale=None, vscale=None):
    _check(lib().h2o_get_kv_scales(h, _ptr(kscale), _ptr(vscale)))


def h2o_set_kv_scales(h, kscale, vscale):
    _check(lib().h2o_set_kv_scales(h, _ptr(kscale), _ptr(vscale)))


def h2o_set_stream(h, stream):
    _check(lib().h2o_set_stream(h, _stream(stream)))


def h2o_set_decode_split(h, ctas_per_unit):
    _check(lib().h2o_set_decode_split(h, int(ctas_per_unit)))


def h2o_sync(h):
    _check(lib().h2o_sync(h))


def h2o_destroy(h):
    lib().h2o_destroy(h)


def h2o_selftest_wait_timeout(h):
    _check(lib().h2o_selftest_wait_timeout(h))


def h2o_prompt_scores_noalloc(Q, K, batch, heads, T, head_dim, dtype, scale, c, stream=None):
    """Prompt column sums into ``c`` without any device allocation (scratch
    is a fixed array inside the library); see include/h2o.h."""
    _check(lib().h2o_prompt_scores_noalloc(_ptr(Q), _ptr(K), batch, heads, int(T), head_dim, dtype,
                                           float(scale), _ptr(c), _stream(stream)))
