"""GPU parity: the CUDA path through the C ABI against the CPU oracle on the
same seeded inputs, at sizes the oracle finishes in seconds that still span
several tiles, several bulk-copy groups and ragged tails."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

import oracle                                              # noqa: E402
from kv_cache_eviction_h2o_gb300 import workloads as wl    # noqa: E402
from parity import (record, Dev, align_prefill, check_out, check_scores, h2o_lockstep, widen,  # noqa: E402
                    kept_lists, lsh_lockstep)

pytestmark = pytest.mark.gpu


def _rand(seed, U, T, S, d, dtype, key_scale=1.0):
    g = np.random.default_rng(seed)
    f = (lambda x: wl.round_bf16(x)) if dtype == "bf16" else (lambda x: x.astype(np.float32))
    Q = f(g.standard_normal((U, T, d), dtype=np.float32))
    K = f(g.standard_normal((U, T, d), dtype=np.float32) * key_scale)
    V = f(g.standard_normal((U, T, d), dtype=np.float32))
    q = f(g.standard_normal((S, U, d), dtype=np.float32))
    k = f(g.standard_normal((S, U, d), dtype=np.float32) * key_scale)
    v = f(g.standard_normal((S, U, d), dtype=np.float32))
    return Q, K, V, q, k, v


@pytest.mark.parametrize("T", [1, 2, 63, 64, 65, 130, 257])
@pytest.mark.parametrize("dtype,d", [("f32", 64), ("bf16", 128)])
def test_prefill_statistics(T, dtype, d):
    U = 3
    Q, K, V, *_ = _rand(100 + T, U, T, 0, d, dtype, key_scale=2.0)
    scale = 1.0 / np.sqrt(d)
    dev = Dev("h2o", U, d, 16, 8, 8, dtype, scale)
    dev.prefill(Q, K, V)
    m, l, c = dev.stats(T)
    mo, lo, co = oracle.prefill_scores(Q, K, scale)
    np.testing.assert_allclose(m, mo, rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(l, lo, rtol=1e-4)
    check_scores(c, co, "column sums")
    np.testing.assert_allclose(c.sum(axis=1), T, rtol=1e-5)
    dev.close()


@pytest.mark.parametrize("U,T", [(1300, 1), (700, 100), (700, 129), (400, 300), (40, 4100)])
def test_prefill_statistics_persistent_walk(U, T):
    """The tensor-core scorer's persistent grid: more (unit, block) items than
    resident CTAs, so every CTA walks several items (short, ragged and
    longest-walked prompts; 4100 tokens = 33 blocks takes one item per CTA)."""
    Q, K, V, *_ = _rand(900 + T, U, T, 0, 128, "bf16", key_scale=2.0)
    scale = 1.0 / np.sqrt(128)
    dev = Dev("h2o", U, 128, 16, 8, 8, "bf16", scale)
    dev.prefill(Q, K, V)
    m, l, c = dev.stats(T)
    mo, lo, co = oracle.prefill_scores(Q, K, scale)
    np.testing.assert_allclose(m, mo, rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(l, lo, rtol=1e-4)
    check_scores(c, co, "column sums")
    np.testing.assert_allclose(c.sum(axis=1), T, rtol=1e-5)
    dev.close()


def test_tiny_workload_h2o():
    w = wl.WORKLOADS["tiny"]
    g = wl.generate(w)
    dev = Dev("h2o", w.units, w.head_dim, w.budget, w.heavy, w.recent, w.dtype, w.scale)
    dev.prefill(g["Q"], g["K"], g["V"])
    st, c, near0 = align_prefill(dev.state(), g["Q"], g["K"], g["V"], w.budget, w.heavy, w.recent, w.scale)
    s = dev.state()
    assert (s["pos"] == st.pos).all()
    check_scores(s["score"], st.score, "prefill scores")
    near, _ = h2o_lockstep(dev, st, g["q"], g["k"], g["v"], w.prompt, w.recent, w.scale)
    record("tiny lockstep", near_ties=near0 + near)
    dev.close()


@pytest.mark.parametrize("split", [1, 2, 3, 4, 8, 16])
def test_opt67b_units_h2o(split):
    w = wl.WORKLOADS["opt-6.7b"]
    units = list(range(12))
    g = wl.generate(w, units=units, steps=24)
    U = len(units)
    dev = Dev("h2o", U, w.head_dim, w.budget, w.heavy, w.recent, w.dtype, w.scale, split=split)
    dev.prefill(g["Q"], g["K"], g["V"])
    st, c, near0 = align_prefill(dev.state(), g["Q"], g["K"], g["V"], w.budget, w.heavy, w.recent, w.scale)
    s = dev.state()
    assert (s["pos"] == st.pos).all()
    assert (s["K"] == st.K).all()
    check_scores(s["score"], st.score, "prefill scores")
    near, _ = h2o_lockstep(dev, st, g["q"], g["k"], g["v"], w.prompt, w.recent, w.scale, check_every=4)
    record("opt-6.7b lockstep split=%d" % split, near_ties=near0 + near)
    dev.close()


@pytest.mark.parametrize("split", [1, 3, 16])
def test_hashevict_units(split):
    w = wl.WORKLOADS["hashevict-opt-6.7b"]
    units = list(range(10))
    g = wl.generate(w, units=units, steps=24)
    W = g["W"]
    U = len(units)
    dev = Dev("lsh", U, w.head_dim, w.budget, 0, w.recent, w.dtype, w.scale, W=W, split=split)
    dev.prefill(g["Q"], g["K"], g["V"])
    st = oracle.lsh_prefill(g["Q"], g["K"], g["V"], W, w.budget, w.recent)
    s = dev.state()
    assert (s["pos"] == st.pos).all()
    assert (s["code"] == st.code).all()
    assert (s["K"] == st.K).all() and (s["V"] == st.V).all()
    lsh_lockstep(dev, st, g["q"], g["k"], g["v"], W, w.prompt, w.recent, w.scale, check_every=4)
    dev.close()


def test_h2o_one_cta_with_a_budget_near_the_chunk_limit():
    # one CTA per unit holding 1000 slots: every slot of the chunk (past 960,
    # the first 5 x 192) must take part in the score update and the arg-min
    T, B, H, r, d = 1300, 1000, 500, 500, 128
    U, S = 2, 6
    Q, K, V, q, k, v = _rand(77, U, T, S, d, "bf16")
    scale = 1.0 / np.sqrt(d)
    dev = Dev("h2o", U, d, B, H, r, "bf16", scale, split=1)
    dev.prefill(Q, K, V)
    st, _, _ = align_prefill(dev.state(), Q, K, V, B, H, r, scale)
    h2o_lockstep(dev, st, q, k, v, T, r, scale)
    dev.close()


@pytest.mark.parametrize("T,B,H,r", [
    (5, 8, 4, 4),        # prompt shorter than the budget: append phase
    (1, 8, 4, 4),        # single-token prompt
    (40, 8, 0, 8),       # no heavy hitters: sliding window
    (40, 8, 8, 0),       # no recent window
    (40, 1, 0, 1),       # one slot
    (40, 1, 1, 0),
    (70, 33, 17, 16),    # ragged groups and tiles
    (130, 129, 64, 65),
    (1500, 1100, 600, 500),  # budget above one CTA's chunk: split across a cluster
])
@pytest.mark.parametrize("dtype,d", [("f32", 64), ("bf16", 128)])
def test_edge_cases_h2o(T, B, H, r, dtype, d):
    U, S = 3, 12
    Q, K, V, q, k, v = _rand(7 * T + B, U, T, S, d, dtype, key_scale=1.5)
    scale = 1.0 / np.sqrt(d)
    dev = Dev("h2o", U, d, B, H, r, dtype, scale)
    dev.prefill(Q, K, V)
    st, c, _ = align_prefill(dev.state(), Q, K, V, B, H, r, scale)
    h2o_lockstep(dev, st, q, k, v, T, r, scale)
    dev.close()


@pytest.mark.parametrize("T,B,r", [(5, 8, 4), (1, 8, 4), (40, 8, 8), (40, 8, 0), (40, 1, 1), (70, 33, 16),
                                   (300, 100, 2),      # smallest window of the pipelined prompt replay
                                   (400, 250, 60), (700, 500, 250),
                                   (600, 480, 480),    # window = budget: one candidate per step
                                   (300, 129, 3), (600, 384, 64), (700, 512, 200),   # four-warp replay: 2, 3, 4 slots a thread
                                   (1500, 1100, 100)])
@pytest.mark.parametrize("dtype,d", [("f32", 64), ("bf16", 128)])
def test_edge_cases_lsh(T, B, r, dtype, d):
    U, S = 3, 12
    Q, K, V, q, k, v = _rand(11 * T + B, U, T, S, d, dtype)
    W = np.random.default_rng(5).standard_normal((d, 32), dtype=np.float32)
    scale = 1.0 / np.sqrt(d)
    dev = Dev("lsh", U, d, B, 0, r, dtype, scale, W=W)
    dev.prefill(Q, K, V)
    st = oracle.lsh_prefill(Q, K, V, W, B, r)
    s = dev.state()
    assert (s["pos"] == st.pos).all() and (s["code"] == st.code).all()
    lsh_lockstep(dev, st, q, k, v, W, T, r, scale)
    dev.close()


def test_full_attention_when_budget_covers_sequence():
    # budget >= prompt + steps: nothing is evicted and every output is full
    # causal attention over all tokens so far
    U, T, S, d = 2, 50, 20, 128
    Q, K, V, q, k, v = _rand(3, U, T, S, d, "bf16")
    scale = 1.0 / np.sqrt(d)
    dev = Dev("h2o", U, d, T + S, 30, T + S - 30, "bf16", scale)
    dev.prefill(Q, K, V)
    for t in range(S):
        out, vic = dev.step(q[t], k[t], v[t])
        assert (vic == -1).all()
        for u in range(U):
            Ka = np.concatenate([K[u], k[: t + 1, u]]).astype(np.float64)
            Va = np.concatenate([V[u], v[: t + 1, u]]).astype(np.float64)
            z = scale * Ka @ q[t, u].astype(np.float64)
            e = np.exp(z - z.max())
            check_out(out[u:u + 1], ((e / e.sum()) @ Va)[None], "full attention")
    dev.close()


def test_state_roundtrip_and_errors():
    from kv_cache_eviction_h2o_gb300 import binding as L
    U, T, d = 2, 30, 64
    Q, K, V, q, k, v = _rand(9, U, T, 3, d, "f32")
    dev = Dev("h2o", U, d, 10, 5, 5, "f32", 0.125)
    # decode before prefill is a state error
    qd = torch.zeros((U, d), device="cuda")
    with pytest.raises(L.H2OError) as e:
        L.h2o_decode_step(dev.h, qd, qd, qd, dev.out, None)
    assert e.value.code == L.H2O_ERR_STATE
    # lsh call on an H2O handle
    dev.prefill(Q, K, V)
    with pytest.raises(L.H2OError) as e:
        L.lsh_decode_step(dev.h, qd, qd, qd, dev.out, None)
    assert e.value.code == L.H2O_ERR_STATE
    s = dev.state()
    dev2 = Dev("h2o", U, d, 10, 5, 5, "f32", 0.125)
    Kh = s["K"].astype(np.float32); Vh = s["V"].astype(np.float32)
    L.h2o_set_state(dev2.h, Kh, Vh, s["score"], s["pos"], None, s["occ"], s["npos"])
    o1, v1 = dev.step(q[0], k[0], v[0])
    o2, v2 = dev2.step(q[0], k[0], v[0])
    assert (v1 == v2).all()
    np.testing.assert_array_equal(o1, o2)
    dev.close(); dev2.close()


@pytest.mark.parametrize("B", [16384, 9217])
def test_largest_budgets_from_a_set_state(B):
    """The largest budget the decode kernels take (16 CTAs of 1024 slots per
    unit, a cluster of 16) and a ragged one (9 full CTAs and one slot more):
    a full cache is written with h2o_set_state -- H heavy positions drawn
    below the window, the recent window, scores and rows random -- and the
    device and the oracle step from that same state."""
    from kv_cache_eviction_h2o_gb300 import binding as L
    U, d, S = 2, 128, 6
    H = B // 2
    r = B - H
    T0 = 3 * B                                   # the position of the first decode step
    rng = np.random.default_rng(B)
    scale = 1.0 / np.sqrt(d)
    st = oracle.H2OState(U, B, d)
    bits = lambda x: (x.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    Kb = bits(wl.round_bf16(rng.standard_normal((U, B, d), dtype=np.float32)))
    Vb = bits(wl.round_bf16(rng.standard_normal((U, B, d), dtype=np.float32)))
    for u in range(U):
        heavy = np.sort(rng.choice(T0 - r, size=H, replace=False))
        st.pos[u] = np.concatenate([heavy, np.arange(T0 - r, T0)]).astype(np.int32)
        st.score[u] = np.where(st.pos[u] < T0 - r, rng.uniform(0.5, 3.0, B), rng.uniform(0.0, 1.0, B))
        # scores exactly representable as the device's fp32 pair
        st.score[u] = st.score[u].astype(np.float32).astype(np.float64)
    st.K = widen(Kb, "bf16").astype(np.float64)
    st.V = widen(Vb, "bf16").astype(np.float64)
    st.occ[:] = B
    dev = Dev("h2o", U, d, B, H, r, "bf16", scale)
    try:
        L.h2o_set_state(dev.h, Kb, Vb, st.score.copy(), st.pos.copy(), None, np.full(U, B, np.int32),
                        np.full(U, T0, np.int32))
        f = lambda *shape: wl.round_bf16(rng.standard_normal(shape, dtype=np.float32))
        q, k, v = f(S, U, d), f(S, U, d), f(S, U, d)
        near, _ = h2o_lockstep(dev, st, q, k, v, T0, r, scale)
        record("largest budget %d" % B, near_ties=near)
    finally:
        dev.close()


def test_largest_budget_hashevict_from_a_set_state():
    """HashEvict at the largest budget (16384 slots, a cluster of 16 CTAs per
    unit): a full cache with random rows, the codes of its keys (the
    oracle's hash) and positions, set on the device; victims, codes,
    positions and rows bit-exact and outputs within tolerance, step by step."""
    from kv_cache_eviction_h2o_gb300 import binding as L
    U, d, S, B = 2, 128, 6, 16384
    r = B // 2
    T0 = 3 * B
    rng = np.random.default_rng(77)
    scale = 1.0 / np.sqrt(d)
    W = np.random.default_rng(5).standard_normal((d, 32), dtype=np.float32)
    st = oracle.LSHState(U, B, d)
    bits = lambda x: (x.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    Kf = wl.round_bf16(rng.standard_normal((U, B, d), dtype=np.float32))
    Vf = wl.round_bf16(rng.standard_normal((U, B, d), dtype=np.float32))
    for u in range(U):
        older = np.sort(rng.choice(T0 - r, size=B - r, replace=False))
        st.pos[u] = np.concatenate([older, np.arange(T0 - r, T0)]).astype(np.int32)
    st.K, st.V = Kf.astype(np.float64), Vf.astype(np.float64)
    st.code = oracle.lsh_codes(Kf, W)
    st.occ[:] = B
    dev = Dev("lsh", U, d, B, 0, r, "bf16", scale, W=W)
    try:
        L.h2o_set_state(dev.h, bits(Kf), bits(Vf), np.zeros((U, B)), st.pos.copy(), st.code.copy(),
                        np.full(U, B, np.int32), np.full(U, T0, np.int32))
        f = lambda *shape: wl.round_bf16(rng.standard_normal(shape, dtype=np.float32))
        q, k, v = f(S, U, d), f(S, U, d), f(S, U, d)
        lsh_lockstep(dev, st, q, k, v, W, T0, r, scale)
    finally:
        dev.close()
