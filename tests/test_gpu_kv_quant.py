"""Quantised cache slots (H2O_KV8, H2O_KV4) on the GPU against the oracle.

Every stored row is int8 or 4-bit codes with one fp32 scale (the quantisers
the oracle defines: amax / 127 or amax / 7, codes rint(x * 127 / amax) or
rint(7 / amax * x) in fp32, half to even; 4-bit codes packed two per byte in
offset binary); a step attends to its own new token at full precision and
stores it quantised.
Codes, scales, positions and victims are compared bit-exactly (H2O victims
up to the counted near ties), outputs and scores within the usual
tolerances.  (H2O: Heavy-Hitter Oracle decode rule; HashEvict: Hamming
replacement rule; the quantised cache is the reading of the Scissorhands
abstract's quantised budgeted cache.)"""
import numpy as np
import pytest

import oracle
from kv_cache_eviction_h2o_gb300 import binding as L
from kv_cache_eviction_h2o_gb300 import workloads as wl
from parity import (Dev, align_prefill, check_scores, h2o_lockstep, lsh_lockstep, record, rows_equal)

pytestmark = pytest.mark.gpu


BITS = [8, 4]


def _quant(st, bits):
    return oracle.kv8(st, bits)


def _h2o_run(w, units, steps, split=0, zero_rows=False, bits=8):
    g = wl.generate(w, units=units, steps=steps)
    if zero_rows:
        # rows with nothing to scale: prompt key/value rows and decode rows of zeros
        g["K"][:, 3] = 0.0; g["V"][:, 5] = 0.0; g["K"][:, -1] = 0.0
        g["k"][2] = 0.0; g["v"][4] = 0.0
    U = len(units)
    dev = Dev("h2o", U, w.head_dim, w.budget, w.heavy, w.recent, w.dtype, w.scale, split=split,
              kv8=bits == 8, kv4=bits == 4)
    dev.prefill(g["Q"], g["K"], g["V"])
    s = dev.state()
    st, c, near0 = align_prefill(s, g["Q"], g["K"], g["V"], w.budget, w.heavy, w.recent, w.scale)
    st = _quant(st, bits)
    assert (s["pos"] == st.pos).all()
    assert rows_equal(s, st), "prompt cache rows differ"
    check_scores(s["score"], st.score, "prefill scores")
    near, _ = h2o_lockstep(dev, st, g["q"], g["k"], g["v"], w.prompt, w.recent, w.scale, check_every=2)
    dev.close()
    return near0, near


@pytest.mark.parametrize("bits", BITS)
def test_quant_tiny_h2o(bits):
    w = wl.WORKLOADS["tiny"]
    _h2o_run(w, list(range(w.units)), w.steps, bits=bits)


@pytest.mark.parametrize("bits", BITS)
@pytest.mark.parametrize("split", [1, 3])
def test_quant_opt67b_units_h2o(split, bits):
    _h2o_run(wl.WORKLOADS["opt-6.7b"], list(range(12)), 24, split=split, bits=bits)


@pytest.mark.parametrize("bits", BITS)
def test_quant_opt67b_many_units_h2o(bits):
    # more units than SMs: one CTA per unit, the many-units tile
    near0, near = _h2o_run(wl.WORKLOADS["opt-6.7b"], list(range(160)), 6, bits=bits)
    record("quant%d opt-6.7b 160 units" % bits, near_ties=near0 + near, sampled_units=160)


@pytest.mark.parametrize("bits", BITS)
def test_quant_zero_rows_h2o(bits):
    _h2o_run(wl.WORKLOADS["tiny"], list(range(4)), 12, zero_rows=True, bits=bits)


@pytest.mark.parametrize("bits", BITS)
@pytest.mark.parametrize("split", [1, 3])
def test_quant_hashevict_units(split, bits):
    w = wl.WORKLOADS["hashevict-opt-6.7b"]
    units = list(range(10))
    g = wl.generate(w, units=units, steps=24)
    W = g["W"]
    dev = Dev("lsh", len(units), w.head_dim, w.budget, 0, w.recent, w.dtype, w.scale, W=W, split=split,
              kv8=bits == 8, kv4=bits == 4)
    dev.prefill(g["Q"], g["K"], g["V"])
    st = _quant(oracle.lsh_prefill(g["Q"], g["K"], g["V"], W, w.budget, w.recent), bits)
    s = dev.state()
    assert (s["pos"] == st.pos).all() and (s["code"] == st.code).all()
    assert rows_equal(s, st)
    lsh_lockstep(dev, st, g["q"], g["k"], g["v"], W, w.prompt, w.recent, w.scale, check_every=2)
    dev.close()


@pytest.mark.parametrize("kind,T,B,H,r", [
    ("h2o", 5, 8, 4, 4),       # prompt shorter than the budget: append phase
    ("h2o", 40, 8, 0, 8),      # sliding window
    ("h2o", 70, 33, 17, 16),   # ragged stage and odd scale rows
    ("lsh", 40, 8, 0, 8),
    ("lsh", 70, 33, 0, 16),
])
@pytest.mark.parametrize("dtype,d", [("f32", 64), ("bf16", 128), ("f32", 128), ("bf16", 64)])
@pytest.mark.parametrize("bits", BITS)
def test_quant_edge_cases(kind, T, B, H, r, dtype, d, bits):
    rng = np.random.default_rng(7 * T + B)
    U, S = 3, 10
    def draw(*shape):
        x = rng.standard_normal(shape).astype(np.float32)
        return wl.round_bf16(x) if dtype == "bf16" else x
    Q, K, V = draw(U, T, d), draw(U, T, d), draw(U, T, d)
    q, k, v = draw(S, U, d), draw(S, U, d), draw(S, U, d)
    scale = 1.0 / np.sqrt(d)
    if kind == "h2o":
        dev = Dev("h2o", U, d, B, H, r, dtype, scale, kv8=bits == 8, kv4=bits == 4)
        dev.prefill(Q, K, V)
        s = dev.state()
        st, _, _ = align_prefill(s, Q, K, V, B, H, r, scale)
        st = _quant(st, bits)
        assert rows_equal(s, st)
        h2o_lockstep(dev, st, q, k, v, T, r, scale)
    else:
        W = np.random.default_rng(5).standard_normal((d, 32), dtype=np.float32)
        dev = Dev("lsh", U, d, B, 0, r, dtype, scale, W=W, kv8=bits == 8, kv4=bits == 4)
        dev.prefill(Q, K, V)
        st = _quant(oracle.lsh_prefill(Q, K, V, W, B, r), bits)
        s = dev.state()
        assert (s["pos"] == st.pos).all() and rows_equal(s, st)
        lsh_lockstep(dev, st, q, k, v, W, T, r, scale)
    dev.close()


@pytest.mark.parametrize("flag", ["H2O_KV8", "H2O_KV4"])
def test_quant_scale_calls(flag):
    h = L.h2o_init(8, 4, 4, 1, 2, 64, L.H2O_F32, 0.125, None)
    ks = np.zeros((2, 8), np.float32)
    with pytest.raises(L.H2OError) as e:
        L.h2o_get_kv_scales(h, ks, ks)
    assert e.value.code == L.H2O_ERR_STATE
    L.h2o_destroy(h)
    h = L.h2o_init(8, 4, 4, 1, 2, 64, L.H2O_F32 | getattr(L, flag), 0.125, None)
    a = np.arange(16, dtype=np.float32).reshape(2, 8) / 7
    b = -a
    L.h2o_set_kv_scales(h, a, b)
    x = np.empty_like(a); y = np.empty_like(b)
    L.h2o_get_kv_scales(h, x, y)
    assert (x == a).all() and (y == b).all()
    with pytest.raises(L.H2OError):
        L.h2o_set_kv_scales(h, a, None)
    L.h2o_destroy(h)


def test_kv4_and_kv8_together_rejected():
    with pytest.raises(L.H2OError) as e:
        L.h2o_init(8, 4, 4, 1, 2, 64, L.H2O_F32 | L.H2O_KV8 | L.H2O_KV4, 0.125, None)
    assert e.value.code == L.H2O_ERR_ARG


@pytest.mark.parametrize("bits", BITS)
def test_quant_largest_budget_from_a_set_state(bits):
    """Quantised slots at the largest budget (16384 slots, a 16-CTA cluster
    per unit): a full cache of random rows quantised by the oracle, its codes,
    scales, positions and scores set on the device; the two step from that
    same state."""
    U, d, S, B = 2, 128, 6, 16384
    H = B // 2
    r = B - H
    T0 = 3 * B
    rng = np.random.default_rng(300 + bits)
    scale = 1.0 / np.sqrt(d)
    st = oracle.H2OState(U, B, d)
    st.K = wl.round_bf16(rng.standard_normal((U, B, d), dtype=np.float32)).astype(np.float64)
    st.V = wl.round_bf16(rng.standard_normal((U, B, d), dtype=np.float32)).astype(np.float64)
    for u in range(U):
        heavy = np.sort(rng.choice(T0 - r, size=H, replace=False))
        st.pos[u] = np.concatenate([heavy, np.arange(T0 - r, T0)]).astype(np.int32)
        st.score[u] = np.where(st.pos[u] < T0 - r, rng.uniform(0.5, 3.0, B), rng.uniform(0.0, 1.0, B))
        st.score[u] = st.score[u].astype(np.float32).astype(np.float64)
    st.occ[:] = B
    st = _quant(st, bits)
    kc, vc = (st.kq, st.vq) if bits == 8 else (oracle.pack4(st.kq), oracle.pack4(st.vq))
    dev = Dev("h2o", U, d, B, H, r, "bf16", scale, kv8=bits == 8, kv4=bits == 4)
    try:
        L.h2o_set_state(dev.h, np.ascontiguousarray(kc), np.ascontiguousarray(vc), st.score.copy(), st.pos.copy(),
                        None, np.full(U, B, np.int32), np.full(U, T0, np.int32))
        L.h2o_set_kv_scales(dev.h, st.ks.copy(), st.vs.copy())
        f = lambda *shape: wl.round_bf16(rng.standard_normal(shape, dtype=np.float32))
        q, k, v = f(S, U, d), f(S, U, d), f(S, U, d)
        near, _ = h2o_lockstep(dev, st, q, k, v, T0, r, scale)
        record("quant%d largest budget" % bits, near_ties=near)
    finally:
        dev.close()
