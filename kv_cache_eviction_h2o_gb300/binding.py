"""Thin ctypes binding of ``libh2o_gb300.so`` with the C ABI's names.

Argument marshalling only: every device-memory argument is a raw pointer
(an ``int``) or any object with ``data_ptr()`` (a torch tensor), every host
buffer of the state calls is a numpy array, and streams are ``cudaStream_t``
values (``int``) or objects with a ``cuda_stream`` attribute.  All compute
runs in the library; a failing call raises ``H2OError`` with the library's
message.  Importing this module does not load the library; the first call
does, and raises if the library was not built (there is no fallback).

The binding remembers each handle's shape (units, budget, head_dim, element
type, query heads per unit, last prompt length) from the calls that made it,
and checks the type and size of every host array, and of every tensor it
is given, before the library writes into or reads from it; a raw integer
pointer is passed through unchecked.
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
H2O_KV4 = 4

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
    "fg_init": (_i, [ctypes.POINTER(_vp), _i, _i, _i, _i, _d, _i, _i, _i, _i, _d, _vp]),
    "fg_prefill": (_i, [_vp, _vp, _vp, _vp, _i]),
    "fg_decode_step": (_i, [_vp, _vp, _vp, _vp, _vp, _vp]),
    "fg_get_policy": (_i, [_vp, _vp, _vp, _vp]),
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


# handle -> its shape, recorded by the init calls
_meta = {}


def _remember(h, kind, U, B, d, dtype, G=1):
    kv8, kv4 = bool(dtype & H2O_KV8), bool(dtype & H2O_KV4)
    elem = np.int8 if kv8 else np.uint8 if kv4 else (np.uint16 if (dtype & H2O_BF16) else np.float32)
    # elements of one stored row: a 4-bit row packs two codes per byte
    _meta[h] = dict(kind=kind, U=U, B=B, d=d, G=G, elem=np.dtype(elem), row=d // 2 if kv4 else d,
                    kv8=kv8, kv4=kv4, T=0, in_size=2 if dtype & H2O_BF16 else 4)
    return h


def _info(h):
    m = _meta.get(h)
    if m is None:
        raise ValueError("unknown handle %r (not created by this binding, or destroyed)" % (h,))
    return m


def _host(x, dtype, n, what):
    """x is None or a C-contiguous numpy array of `dtype` with n elements."""
    if x is None:
        return None
    if not isinstance(x, np.ndarray):
        raise TypeError("%s must be a numpy array (host memory)" % what)
    if x.dtype != np.dtype(dtype):
        raise TypeError("%s must have dtype %s (got %s)" % (what, np.dtype(dtype), x.dtype))
    if x.size != n:
        raise ValueError("%s must have %d elements (got %d)" % (what, n, x.size))
    if not x.flags["C_CONTIGUOUS"]:
        raise ValueError("%s must be C-contiguous" % what)
    return x


def _dev(x, nbytes, what, dtypes=None):
    """Check a device tensor's size (and dtype) when it is one; raw integer
    pointers pass unchecked."""
    if x is None or isinstance(x, int) or not hasattr(x, "numel"):
        return x
    if getattr(x, "device", None) is not None and getattr(x.device, "type", "cuda") != "cuda":
        raise ValueError("%s must be on the GPU" % what)
    got = x.numel() * x.element_size()
    if got < nbytes:
        raise ValueError("%s holds %d bytes, needs %d" % (what, got, nbytes))
    if dtypes is not None and str(x.dtype).replace("torch.", "") not in dtypes:
        raise TypeError("%s must be of dtype %s (got %s)" % (what, "/".join(dtypes), x.dtype))
    return x


def h2o_last_error():
    return lib().h2o_last_error().decode()


def h2o_init(budget, heavy, recent, batch, heads, head_dim, dtype, scale, stream=None):
    h = _vp()
    _check(lib().h2o_init(ctypes.byref(h), budget, heavy, recent, batch, heads, head_dim, dtype,
                          float(scale), _stream(stream)))
    return _remember(h.value, "h2o", batch * heads, budget, head_dim, dtype)


def h2o_init_gqa(budget, heavy, recent, batch, kv_heads, groups, head_dim, dtype, scale, stream=None):
    h = _vp()
    _check(lib().h2o_init_gqa(ctypes.byref(h), budget, heavy, recent, batch, kv_heads, groups, head_dim,
                              dtype, float(scale), _stream(stream)))
    return _remember(h.value, "h2o", batch * kv_heads, budget, head_dim, dtype, groups)


def lsh_init(budget, recent, batch, heads, head_dim, dtype, scale, W, stream=None):
    h = _vp()
    _dev(W, head_dim * 32 * 4, "W", ("float32",))
    _check(lib().lsh_init(ctypes.byref(h), budget, recent, batch, heads, head_dim, dtype, float(scale),
                          _ptr(W), _stream(stream)))
    return _remember(h.value, "lsh", batch * heads, budget, head_dim, dtype)


def h2o_prefill(h, Q, K, V, T):
    _prompt_args(h, Q, K, V, T)
    _check(lib().h2o_prefill(h, _ptr(Q), _ptr(K), _ptr(V), int(T)))
    _info(h)["T"] = int(T)


def lsh_prefill(h, Q, K, V, T):
    _prompt_args(h, Q, K, V, T)
    _check(lib().lsh_prefill(h, _ptr(Q), _ptr(K), _ptr(V), int(T)))
    _info(h)["T"] = int(T)


def h2o_decode_step(h, q, k, v, out, victim_out=None):
    _step_args(h, q, k, v, out, victim_out)
    _check(lib().h2o_decode_step(h, _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(victim_out)))


def lsh_decode_step(h, q, k, v, out, victim_out=None):
    _step_args(h, q, k, v, out, victim_out)
    _check(lib().lsh_decode_step(h, _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(victim_out)))


def sh_init(budget, heavy, recent, batch, heads, head_dim, dtype, scale, stream=None):
    h = _vp()
    _check(lib().sh_init(ctypes.byref(h), budget, heavy, recent, batch, heads, head_dim, dtype,
                         float(scale), _stream(stream)))
    return _remember(h.value, "sh", batch * heads, budget, head_dim, dtype)


def sh_prefill(h, Q, K, V, T):
    _prompt_args(h, Q, K, V, T)
    _check(lib().sh_prefill(h, _ptr(Q), _ptr(K), _ptr(V), int(T)))
    _info(h)["T"] = int(T)


def sh_decode_step(h, q, k, v, out, victim_out=None):
    _step_args(h, q, k, v, out, victim_out)
    _check(lib().sh_decode_step(h, _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(victim_out)))


def _prompt_args(h, Q, K, V, T):
    m = _info(h)
    row = m["d"] * m["in_size"]
    _dev(Q, m["U"] * m["G"] * int(T) * row, "Q")
    _dev(K, m["U"] * int(T) * row, "K")
    _dev(V, m["U"] * int(T) * row, "V")


def _step_args(h, q, k, v, out, victim_out):
    m = _info(h)
    row = m["d"] * m["in_size"]
    _dev(q, m["U"] * m["G"] * row, "q")
    _dev(k, m["U"] * row, "k")
    _dev(v, m["U"] * row, "v")
    _dev(out, m["U"] * m["G"] * m["d"] * 4, "out", ("float32",))
    _dev(victim_out, m["U"] * 4, "victim_out", ("int32",))


def _state_args(h, K, V, score, pos, code, occupancy, next_pos):
    m = _info(h)
    UB = m["U"] * m["B"]
    _host(K, m["elem"], UB * m["row"], "K")
    _host(V, m["elem"], UB * m["row"], "V")
    _host(score, np.float64, UB, "score")
    _host(pos, np.int32, UB, "pos")
    _host(code, np.uint32, UB, "code")
    _host(occupancy, np.int32, m["U"], "occupancy")
    _host(next_pos, np.int32, m["U"], "next_pos")


def fg_init(budget, heavy, recent, full_budget, tau, batch, heads, head_dim, dtype, scale, stream=None):
    h = _vp()
    _check(lib().fg_init(ctypes.byref(h), budget, heavy, recent, full_budget, float(tau), batch, heads, head_dim,
                         dtype, float(scale), _stream(stream)))
    return _remember(h.value, "fg", batch * heads, max(budget, full_budget), head_dim, dtype)


def fg_prefill(h, Q, K, V, T):
    _prompt_args(h, Q, K, V, T)
    _check(lib().fg_prefill(h, _ptr(Q), _ptr(K), _ptr(V), int(T)))
    _info(h)["T"] = int(T)


def fg_decode_step(h, q, k, v, out, victim_out=None):
    _step_args(h, q, k, v, out, victim_out)
    _check(lib().fg_decode_step(h, _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(victim_out)))


def fg_get_policy(h, policy=None, rec_local=None, rec_freq=None):
    U = _info(h)["U"]
    _host(policy, np.int32, U, "policy")
    _host(rec_local, np.float64, U, "rec_local")
    _host(rec_freq, np.float64, U, "rec_freq")
    _check(lib().fg_get_policy(h, _ptr(policy), _ptr(rec_local), _ptr(rec_freq)))


def h2o_get_state(h, K=None, V=None, score=None, pos=None, code=None, occupancy=None, next_pos=None):
    _state_args(h, K, V, score, pos, code, occupancy, next_pos)
    _check(lib().h2o_get_state(h, _ptr(K), _ptr(V), _ptr(score), _ptr(pos), _ptr(code), _ptr(occupancy),
                               _ptr(next_pos)))


def h2o_set_state(h, K=None, V=None, score=None, pos=None, code=None, occupancy=None, next_pos=None):
    _state_args(h, K, V, score, pos, code, occupancy, next_pos)
    _check(lib().h2o_set_state(h, _ptr(K), _ptr(V), _ptr(score), _ptr(pos), _ptr(code), _ptr(occupancy),
                               _ptr(next_pos)))


def h2o_get_prefill_stats(h, m=None, l=None, c=None):
    i = _info(h)
    n = i["U"] * i["T"]
    _host(m, np.float32, n * i["G"], "m")
    _host(l, np.float32, n * i["G"], "l")
    _host(c, np.float64, n, "c")
    _check(lib().h2o_get_prefill_stats(h, _ptr(m), _ptr(l), _ptr(c)))


def h2o_get_kv_scales(h, kscale=None, vscale=None):
    i = _info(h)
    _host(kscale, np.float32, i["U"] * i["B"], "kscale")
    _host(vscale, np.float32, i["U"] * i["B"], "vscale")
    _check(lib().h2o_get_kv_scales(h, _ptr(kscale), _ptr(vscale)))


def h2o_set_kv_scales(h, kscale, vscale):
    i = _info(h)
    _host(kscale, np.float32, i["U"] * i["B"], "kscale")
    _host(vscale, np.float32, i["U"] * i["B"], "vscale")
    _check(lib().h2o_set_kv_scales(h, _ptr(kscale), _ptr(vscale)))


def h2o_set_stream(h, stream):
    _check(lib().h2o_set_stream(h, _stream(stream)))


def h2o_set_decode_split(h, ctas_per_unit):
    _check(lib().h2o_set_decode_split(h, int(ctas_per_unit)))


def h2o_sync(h):
    _check(lib().h2o_sync(h))


def h2o_destroy(h):
    lib().h2o_destroy(h)
    _meta.pop(h, None)


def h2o_selftest_wait_timeout(h):
    _check(lib().h2o_selftest_wait_timeout(h))


def h2o_prompt_scores_noalloc(Q, K, batch, heads, T, head_dim, dtype, scale, c, stream=None):
    """Prompt column sums into ``c`` without any device allocation (scratch
    is a fixed array inside the library); see include/h2o.h."""
    esz = 2 if dtype & H2O_BF16 else 4
    _dev(Q, batch * heads * int(T) * head_dim * esz, "Q")
    _dev(K, batch * heads * int(T) * head_dim * esz, "K")
    _dev(c, batch * heads * int(T) * 8, "c", ("float64",))
    _check(lib().h2o_prompt_scores_noalloc(_ptr(Q), _ptr(K), batch, heads, int(T), head_dim, dtype,
                                           float(scale), _ptr(c), _stream(stream)))
