"""CPU oracle for budgeted-KV decode attention with H2O heavy-hitter eviction
and the HashEvict LSH variant.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, the package smoke check and
the benchmark's CPU-baseline leg, never by the product path.  The arithmetic
lives in ``oracle.c`` (plain C, fp64); this module only marshals numpy arrays
through ctypes.  Every array is C-contiguous; floating inputs are float64
holding the exact values the device path reads (bf16/fp32 upcast), the LSH
projection matrix is float32.

Shapes use U = batch*heads independent units:
  prompt Q, K, V  [U, T, d]      decode q, k, v  [U, d]
  cache K, V      [U, B, d]      score [U, B]  pos [U, B]  occ [U]
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None

_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_u32p = np.ctypeslib.ndpointer(dtype=np.uint32, flags="C_CONTIGUOUS")
_vp = ctypes.c_void_p
_i = ctypes.c_int
_d = ctypes.c_double


def lib():
    global _lib
    if _lib is None:
        # ORACLE_LIB lets the mutation tests load a deliberately broken copy
        path = os.environ.get("ORACLE_LIB") or _build.build()
        L = ctypes.CDLL(path)
        L.oracle_set_threads.argtypes = [_i]
        L.oracle_get_threads.restype = _i
        L.oracle_prefill_scores.argtypes = [_i, _i, _i, _d, _f64p, _f64p, _f64p, _f64p, _f64p]
        L.oracle_select.argtypes = [_i, _i, _i, _i, _f64p, _i32p, _vp]
        L.oracle_select.restype = _i
        L.oracle_build_cache.argtypes = [_i, _i, _i, _i, _i32p, _i32p, _f64p, _f64p, _f64p,
                                         _f64p, _f64p, _f64p, _i32p, _i32p]
        L.oracle_h2o_prefill.argtypes = [_i, _i, _i, _i, _i, _i, _d, _f64p, _f64p, _f64p,
                                         _f64p, _f64p, _f64p, _i32p, _i32p, _vp, _vp, _vp]
        L.oracle_h2o_decode_step.argtypes = [_i, _i, _i, _i, _d, _i, _f64p, _f64p, _f64p,
                                             _i32p, _i32p, _f64p, _f64p, _f64p, _f64p,
                                             _vp, _vp, _vp, _vp]
        L.oracle_quantize_rows.argtypes = [_i, _i, _f64p, _vp, _f32p]
        L.oracle_quantize_rows4.argtypes = [_i, _i, _f64p, _vp, _f32p]
        L.oracle_h2o_decode_step_gqa.argtypes = [_i, _i, _i, _i, _i, _d, _i, _f64p, _f64p, _f64p,
                                                 _i32p, _i32p, _f64p, _f64p, _f64p, _f64p,
                                                 _vp, _vp, _vp, _vp]
        L.oracle_lsh_code.argtypes = [_i, _f64p, _f32p]
        L.oracle_lsh_code.restype = ctypes.c_uint32
        L.oracle_lsh_codes.argtypes = [_i, _i, _f64p, _f32p, _u32p]
        L.oracle_lsh_prefill.argtypes = [_i, _i, _i, _i, _i, _f64p, _f64p, _f64p, _f32p,
                                         _f64p, _f64p, _u32p, _i32p, _i32p]
        L.oracle_lsh_decode_step.argtypes = [_i, _i, _i, _i, _d, _i, _f64p, _f64p, _u32p,
                                             _i32p, _i32p, _f64p, _f64p, _f64p, _f32p,
                                             _f64p, _vp]
        L.oracle_sh_prompt_masks.argtypes = [_i, _i, _i, _d, _f64p, _f64p, _u32p, _f64p, _vp]
        L.oracle_sh_select.argtypes = [_i, _i, _i, _i, _u32p, _i32p]
        L.oracle_sh_select.restype = _i
        L.oracle_sh_decode_step.argtypes = [_i, _i, _i, _i, _d, _i, _f64p, _f64p, _u32p,
                                            _i32p, _i32p, _f64p, _f64p, _f64p, _f64p,
                                            _vp, _vp, _vp, _vp]
        L.oracle_fg_profile.argtypes = [_i, _i, _i, _i, _i, _i, _d, _d, _f64p, _f64p, _i32p, _f64p, _f64p]
        _lib = L
    return _lib


def _c64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def set_threads(n: int) -> None:
    lib().oracle_set_threads(int(n))


def get_threads() -> int:
    return int(lib().oracle_get_threads())


def prefill_scores(Q, K, scale):
    """Row max m, row normaliser l and column sums c of the causal prompt
    softmax, each [U, T] float64."""
    Q = _c64(Q); K = _c64(K)
    U, T, d = Q.shape
    m = np.empty((U, T)); l = np.empty((U, T)); c = np.empty((U, T))
    lib().oracle_prefill_scores(U, T, d, float(scale), Q, K, m, l, c)
    return m, l, c


def select(c, B, H, r):
    """Kept prompt positions (ascending) for one unit and the relative
    score gap at the heavy-hitter cut (inf when no choice was made)."""
    c = _c64(c)
    T = c.shape[0]
    kept = np.empty(max(T, 1), dtype=np.int32)
    margin = np.empty(1)
    n = lib().oracle_select(T, B, H, r, c, kept, _ptr(margin))
    return kept[:n].copy(), float(margin[0])


class H2OState:
    """Oracle H2O cache for U units (all arrays float64 / int32)."""

    def __init__(self, U, B, d):
        self.U, self.B, self.d = U, B, d
        self.K = np.zeros((U, B, d))
        self.V = np.zeros((U, B, d))
        self.score = np.zeros((U, B))
        self.pos = np.full((U, B), -1, dtype=np.int32)
        self.occ = np.zeros(U, dtype=np.int32)

    def copy(self):
        s = H2OState(self.U, self.B, self.d)
        for name in ("K", "V", "score", "pos", "occ", "kq", "ks", "vq", "vs"):
            if hasattr(self, name):
                setattr(s, name, getattr(self, name).copy())
        if hasattr(self, "qbits"):
            s.qbits = self.qbits
        return s


def h2o_prefill(Q, K, V, B, H, r, scale):
    """Prompt phase: returns (state, c [U,T], kept [U,B] (-1 padded),
    margin [U])."""
    Q = _c64(Q); K = _c64(K); V = _c64(V)
    U, T, d = Q.shape
    st = H2OState(U, B, d)
    c = np.empty((U, T))
    kept = np.empty((U, B), dtype=np.int32)
    margin = np.empty(U)
    lib().oracle_h2o_prefill(U, T, d, B, H, r, float(scale), Q, K, V,
                             st.K, st.V, st.score, st.pos, st.occ,
                             _ptr(c), _ptr(kept), _ptr(margin))
    return st, c, kept, margin


def build_cache(K, V, c, kept, B):
    """Cache built from explicit kept lists ([U, B], -1 padded, ascending)."""
    K = _c64(K); V = _c64(V); c = _c64(c)
    U, T, d = K.shape
    kept = np.ascontiguousarray(kept, dtype=np.int32)
    nkept = np.ascontiguousarray((kept >= 0).sum(axis=1), dtype=np.int32)
    st = H2OState(U, B, d)
    lib().oracle_build_cache(U, T, d, B, kept, nkept, c, K, V,
                             st.K, st.V, st.score, st.pos, st.occ)
    return st


def h2o_decode_step(st, q, k, v, p, r, scale, forced=None):
    """One decode step in place on ``st``.  Returns (out [U,d], victim [U],
    margin [U], evicted [U])."""
    q = _c64(q); k = _c64(k); v = _c64(v)
    U, d = q.shape
    out = np.empty((U, d))
    victim = np.empty(U, dtype=np.int32)
    margin = np.empty(U)
    evicted = np.empty(U)
    f = None if forced is None else np.ascontiguousarray(forced, dtype=np.int32)
    lib().oracle_h2o_decode_step(U, d, st.B, r, float(scale), int(p), st.K, st.V,
                                 st.score, st.pos, st.occ, q, k, v, out,
                                 _ptr(victim), _ptr(margin), _ptr(evicted), _ptr(f))
    if hasattr(st, "kq"):
        # int8 cache: the step attended to the new token at full precision;
        # the slot it now occupies stores the quantised row
        _kv8_written(st, _written_slots(victim, st.occ))
    return out, victim, margin, evicted


def quantize_rows(X, bits=8):
    """int8 (bits 8, codes within +-127) or 4-bit (bits 4, codes within
    +-7, one per byte) codes [..., d] and fp32 scales [...] of every row of
    X (values exactly representable in fp32)."""
    X = _c64(X)
    flat = X.reshape(-1, X.shape[-1])
    code = np.empty(flat.shape, dtype=np.int8)
    scale = np.empty(flat.shape[0], dtype=np.float32)
    fn = lib().oracle_quantize_rows if bits == 8 else lib().oracle_quantize_rows4
    fn(flat.shape[0], flat.shape[1], flat, code.ctypes.data_as(ctypes.c_void_p), scale)
    return code.reshape(X.shape), scale.reshape(X.shape[:-1])


def pack4(code):
    """4-bit codes [..., d] (one per byte, within +-7) packed two per byte
    [..., d/2] in offset binary: each nibble holds code + 8 (1..15), element
    2i in the low nibble and 2i+1 in the high one."""
    c = (np.asarray(code, np.int16) + 8).astype(np.uint8)
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def dequantize(code, scale):
    """code * scale, exactly, as float64."""
    return code.astype(np.float64) * scale.astype(np.float64)[..., None]


def kv8(st, bits=8):
    """Turn a freshly built cache (exact rows) into a quantised cache (int8
    rows, or 4-bit rows with bits=4): every row is quantised, its codes and
    scales kept on the state, and the rows the arithmetic reads become the
    dequantised values."""
    st.qbits = bits
    st.kq, st.ks = quantize_rows(st.K, bits)
    st.vq, st.vs = quantize_rows(st.V, bits)
    st.K = dequantize(st.kq, st.ks)
    st.V = dequantize(st.vq, st.vs)
    return st


def kv4(st):
    """kv8 with 4-bit rows."""
    return kv8(st, 4)


def _kv8_written(st, slots):
    """Quantise the row each unit's step wrote (slots[u], exact values)."""
    bits = getattr(st, "qbits", 8)
    for u, s in enumerate(slots):
        kq, ks = quantize_rows(st.K[u, s][None], bits)
        vq, vs = quantize_rows(st.V[u, s][None], bits)
        st.kq[u, s], st.ks[u, s] = kq[0], ks[0]
        st.vq[u, s], st.vs[u, s] = vq[0], vs[0]
        st.K[u, s] = dequantize(kq, ks)[0]
        st.V[u, s] = dequantize(vq, vs)[0]


def _written_slots(victim, occ_after):
    return [int(v) if v >= 0 else int(o) - 1 for v, o in zip(victim, occ_after)]


def h2o_prefill_gqa(Q, K, V, B, H, r, scale):
    """Prompt phase of a cache shared by G query heads: Q [U*G, T, d] (the
    G heads of cache unit u are rows u*G .. u*G+G-1), K, V [U, T, d].  Each
    head's column sums use its unit's keys; a unit's column sums are the sum
    over its heads (g = 0..G-1); selection and cache as for one head.
    Returns (state, c [U, T], kept [U, B], margin [U], per-head c [U*G, T])."""
    Q = _c64(Q); K = _c64(K); V = _c64(V)
    U, T, d = K.shape
    G = Q.shape[0] // U
    _, _, cq = prefill_scores(Q, np.repeat(K, G, axis=0), scale)
    c = np.zeros((U, T))
    for g in range(G):
        c += cq[g::G]
    kept = np.full((U, B), -1, np.int32)
    margin = np.empty(U)
    for u in range(U):
        ku, margin[u] = select(c[u], B, H, r)
        kept[u, :len(ku)] = ku
    st = build_cache(K, V, c, kept, B)
    return st, c, kept, margin, cq


def h2o_decode_step_gqa(st, q, k, v, p, r, scale, forced=None):
    """One grouped-query decode step in place on ``st``: q [U*G, d] (heads
    of unit u in rows u*G ..), k, v [U, d].  Returns (out [U*G, d], victim
    [U], margin [U], evicted [U])."""
    q = _c64(q); k = _c64(k); v = _c64(v)
    U, d = k.shape
    G = q.shape[0] // U
    out = np.empty((U * G, d))
    victim = np.empty(U, dtype=np.int32)
    margin = np.empty(U)
    evicted = np.empty(U)
    f = None if forced is None else np.ascontiguousarray(forced, dtype=np.int32)
    lib().oracle_h2o_decode_step_gqa(U, G, d, st.B, r, float(scale), int(p), st.K, st.V,
                                     st.score, st.pos, st.occ, q, k, v, out,
                                     _ptr(victim), _ptr(margin), _ptr(evicted), _ptr(f))
    if hasattr(st, "kq"):
        # int8 cache: as for one head, the written slot stores the quantised row
        _kv8_written(st, _written_slots(victim, st.occ))
    return out, victim, margin, evicted


def lsh_code(x, W):
    x = _c64(x)
    W = np.ascontiguousarray(W, dtype=np.float32)
    return int(lib().oracle_lsh_code(x.shape[0], x, W))


def lsh_codes(X, W):
    """Codes of every row of X [..., d] -> uint32 [...]."""
    X = _c64(X)
    W = np.ascontiguousarray(W, dtype=np.float32)
    flat = X.reshape(-1, X.shape[-1])
    out = np.empty(flat.shape[0], dtype=np.uint32)
    lib().oracle_lsh_codes(flat.shape[0], flat.shape[1], flat, W, out)
    return out.reshape(X.shape[:-1])


class LSHState:
    def __init__(self, U, B, d):
        self.U, self.B, self.d = U, B, d
        self.K = np.zeros((U, B, d))
        self.V = np.zeros((U, B, d))
        self.code = np.zeros((U, B), dtype=np.uint32)
        self.pos = np.full((U, B), -1, dtype=np.int32)
        self.occ = np.zeros(U, dtype=np.int32)


def lsh_prefill(Q, K, V, W, B, r):
    Q = _c64(Q); K = _c64(K); V = _c64(V)
    W = np.ascontiguousarray(W, dtype=np.float32)
    U, T, d = Q.shape
    st = LSHState(U, B, d)
    lib().oracle_lsh_prefill(U, T, d, B, r, Q, K, V, W, st.K, st.V, st.code, st.pos, st.occ)
    return st


def lsh_decode_step(st, q, k, v, W, p, r, scale):
    """One HashEvict step in place on ``st``.  Returns (out [U,d], victim [U])."""
    q = _c64(q); k = _c64(k); v = _c64(v)
    W = np.ascontiguousarray(W, dtype=np.float32)
    U, d = q.shape
    out = np.empty((U, d))
    victim = np.empty(U, dtype=np.int32)
    lib().oracle_lsh_decode_step(U, d, st.B, r, float(scale), int(p), st.K, st.V,
                                 st.code, st.pos, st.occ, q, k, v, W, out, _ptr(victim))
    if hasattr(st, "kq"):
        _kv8_written(st, _written_slots(victim, st.occ))
    return out, victim


class SHState:
    """Oracle cache of the persistence-of-importance rule for U units: rows
    (float64), each slot's 32-step pivotal history (uint32, bit 0 = the
    latest step), positions and occupancy."""

    def __init__(self, U, B, d):
        self.U, self.B, self.d = U, B, d
        self.K = np.zeros((U, B, d))
        self.V = np.zeros((U, B, d))
        self.mask = np.zeros((U, B), dtype=np.uint32)
        self.pos = np.full((U, B), -1, dtype=np.int32)
        self.occ = np.zeros(U, dtype=np.int32)

    def copy(self):
        s = SHState(self.U, self.B, self.d)
        for name in ("K", "V", "mask", "pos", "occ"):
            setattr(s, name, getattr(self, name).copy())
        return s


def sh_prompt_masks(Q, K, scale, with_t=False):
    """Pivotal histories of every prompt token after the prompt: [U, T]
    uint32 (bit T-1-i set when the token was pivotal for query row i, over
    the last 32 rows), and the smallest |P * m - 1| among those decisions
    per unit; with_t: also P * m of every decision, [U, 32, T] (window row
    w = row i - max(0, T - 32))."""
    Q = _c64(Q); K = _c64(K)
    U, T, d = Q.shape
    mask = np.empty((U, T), dtype=np.uint32)
    margin = np.empty(U)
    t = np.empty((U, 32, T)) if with_t else None
    lib().oracle_sh_prompt_masks(U, T, d, float(scale), Q, K, mask, margin, _ptr(t))
    return (mask, margin, t) if with_t else (mask, margin)


def sh_build_cache(K, V, mask, kept, B):
    """Cache from explicit kept lists ([U, B] ascending positions, -1
    padded): slot s holds kept position s with that token's history."""
    K = _c64(K); V = _c64(V)
    U, T, d = K.shape
    st = SHState(U, B, d)
    for u in range(U):
        ks = kept[u][kept[u] >= 0]
        n = len(ks)
        st.K[u, :n] = K[u, ks]
        st.V[u, :n] = V[u, ks]
        st.mask[u, :n] = mask[u, ks]
        st.pos[u, :n] = ks
        st.occ[u] = n
    return st


def sh_prefill(Q, K, V, B, H, r, scale):
    """Prompt phase of the persistence-of-importance cache: returns (state,
    masks [U, T], kept [U, B] (-1 padded), margin [U])."""
    mask, margin = sh_prompt_masks(Q, K, scale)
    U, T = mask.shape
    kept = np.empty((U, B), dtype=np.int32)
    for u in range(U):
        lib().oracle_sh_select(T, B, H, r, np.ascontiguousarray(mask[u]), kept[u])
    return sh_build_cache(K, V, mask, kept, B), mask, kept, margin


def sh_decode_step(st, q, k, v, p, r, scale, forced=None, with_t=False):
    """One decode step in place on ``st``.  Returns (out [U, d], victim [U],
    margin [U]); with_t: also P * m of every decided flag, [U, B+1] (the new
    token at index B)."""
    q = _c64(q); k = _c64(k); v = _c64(v)
    U, d = q.shape
    out = np.empty((U, d))
    victim = np.empty(U, dtype=np.int32)
    margin = np.empty(U)
    t = np.zeros((U, st.B + 1)) if with_t else None
    f = None if forced is None else np.ascontiguousarray(forced, dtype=np.int32)
    lib().oracle_sh_decode_step(U, d, st.B, r, float(scale), int(p), st.K, st.V, st.mask,
                                st.pos, st.occ, q, k, v, out, _ptr(victim), _ptr(margin), _ptr(f), _ptr(t))
    return (out, victim, margin, t) if with_t else (out, victim, margin)


def fg_profile(Q, K, B, H, r, scale, tau):
    """Per-head cache policy from the prompt's attention: (policy [U] int32,
    0 local / 1 frequency + local / 2 full; recovery of local [U]; recovery
    of frequency + local [U])."""
    Q = _c64(Q); K = _c64(K)
    U, T, d = Q.shape
    policy = np.empty(U, dtype=np.int32)
    rl = np.empty(U)
    rf = np.empty(U)
    lib().oracle_fg_profile(U, T, d, B, H, r, float(scale), float(tau), Q, K, policy, rl, rf)
    return policy, rl, rf


def fg_policy_params(policy, B, H, r, B_full):
    """(budget, heavy, recent) of a head's policy: local keeps the newest B
    tokens (no heavy slots, the window is the whole budget), frequency +
    local is the H2O cache (B, H, r), full keeps up to B_full tokens with
    nothing evicted while they fit."""
    return {0: (B, 0, B), 1: (B, H, r), 2: (B_full, 0, B_full)}[int(policy)]


def fg_prefill(Q, K, V, B, H, r, scale, tau, B_full):
    """Per-head policies from the prompt (fg_profile), then each unit's
    cache built by the H2O prompt rule with its policy's parameters.
    Returns (policy [U], per-unit H2OState list, per-unit (B, H, r))."""
    policy, _, _ = fg_profile(Q, K, B, H, r, scale, tau)
    states, params = [], []
    for u in range(Q.shape[0]):
        Bu, Hu, ru = fg_policy_params(policy[u], B, H, r, B_full)
        st, _, _, _ = h2o_prefill(Q[u:u + 1], K[u:u + 1], V[u:u + 1], Bu, Hu, ru, scale)
        states.append(st)
        params.append((Bu, Hu, ru))
    return policy, states, params


def fg_decode_step(states, params, q, k, v, p, scale):
    """One decode step of every unit with its own policy's window.  Returns
    (out [U, d], victim [U])."""
    U, d = q.shape
    out = np.empty((U, d))
    victim = np.empty(U, dtype=np.int32)
    for u in range(U):
        o, vic, _, _ = h2o_decode_step(states[u], q[u:u + 1], k[u:u + 1], v[u:u + 1], p, params[u][2], scale)
        out[u] = o[0]
        victim[u] = vic[0]
    return out, victim
