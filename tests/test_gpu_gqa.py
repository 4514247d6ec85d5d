"""Grouped-query caches (h2o_init_gqa) on the GPU against the oracle.

A cache unit is shared by G query heads: every head attends with its own
softmax; a slot's score grows by the sum of the heads' probabilities, a
prompt token's column sum is the sum over the heads, the new token's score
is the sum of its G own probabilities (the reading of the accumulated
attention of the H2O review page, 提案手法, for a shared slot).  Positions,
victims and cache rows bit-exact (H2O victims up to counted near ties),
outputs and scores within the usual tolerances."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

import oracle                                              # noqa: E402
from kv_cache_eviction_h2o_gb300 import binding as L       # noqa: E402
from kv_cache_eviction_h2o_gb300 import workloads as wl    # noqa: E402
from parity import (record, Dev, align_prefill, check_out, check_scores, h2o_lockstep,  # noqa: E402
                    rows_equal)

pytestmark = pytest.mark.gpu


def _rand(seed, U, G, T, S, d, dtype, key_scale=1.0):
    g = np.random.default_rng(seed)
    f = (lambda x: wl.round_bf16(x)) if dtype == "bf16" else (lambda x: x.astype(np.float32))
    Q = f(g.standard_normal((U * G, T, d), dtype=np.float32))
    K = f(g.standard_normal((U, T, d), dtype=np.float32) * key_scale)
    V = f(g.standard_normal((U, T, d), dtype=np.float32))
    q = f(g.standard_normal((S, U * G, d), dtype=np.float32))
    k = f(g.standard_normal((S, U, d), dtype=np.float32) * key_scale)
    v = f(g.standard_normal((S, U, d), dtype=np.float32))
    return Q, K, V, q, k, v


def _run(U, G, T, B, H, r, S, d, dtype, seed, kv8=False, key_scale=1.5, check_every=1, kv4=False):
    Q, K, V, q, k, v = _rand(seed, U, G, T, S, d, dtype, key_scale)
    scale = 1.0 / np.sqrt(d)
    dev = Dev("h2o", U, d, B, H, r, dtype, scale, kv8=kv8, groups=G, kv4=kv4)
    dev.prefill(Q, K, V)
    s = dev.state()
    st, c, near0 = align_prefill(s, Q, K, V, B, H, r, scale)
    if kv8:
        st = oracle.kv8(st)
    if kv4:
        st = oracle.kv4(st)
    assert (s["pos"] == st.pos).all(), "prompt positions differ"
    assert rows_equal(s, st), "prompt cache rows differ"
    check_scores(s["score"], st.score, "prompt scores")
    near, st = h2o_lockstep(dev, st, q, k, v, T, r, scale, check_every=check_every)
    dev.close()
    return near0, near


@pytest.mark.parametrize("G", [2, 4, 8])
@pytest.mark.parametrize("dtype,d", [("f32", 64), ("bf16", 128)])
def test_gqa_prefill_and_decode(G, dtype, d):
    # 200-slot cache: two rounds of six warps' 16-slot stages, a ragged tail,
    # and each head's CTA updating its share of the scores
    _run(U=3, G=G, T=400, B=200, H=100, r=100, S=10, d=d, dtype=dtype, seed=11 * G + d)


@pytest.mark.parametrize("T,B,H,r", [
    (5, 8, 4, 4),            # append phase
    (1, 8, 4, 4),            # single-token prompt
    (40, 8, 0, 8),           # sliding window
    (40, 8, 8, 0),           # no recent window
    (40, 1, 1, 0),           # one slot
    (70, 33, 17, 16),        # ragged
    (1300, 1024, 512, 512),  # the largest grouped-query budget
])
def test_gqa_edge_cases(T, B, H, r):
    _run(U=2, G=4, T=T, B=B, H=H, r=r, S=8, d=128, dtype="bf16", seed=3 * T + B)


def test_gqa_sixteen_heads_per_unit():
    # the largest group: a 16-CTA cluster per cache unit
    _run(U=2, G=16, T=300, B=120, H=60, r=60, S=6, d=128, dtype="bf16", seed=5)


@pytest.mark.parametrize("G", [1, 4])
def test_gqa_int8_slots(G):
    _run(U=3, G=G, T=400, B=200, H=100, r=100, S=8, d=128, dtype="bf16", seed=21 + G, kv8=True)


@pytest.mark.parametrize("G,dtype,d", [(1, "bf16", 128), (4, "bf16", 128), (2, "f32", 64)])
def test_gqa_4bit_slots(G, dtype, d):
    _run(U=3, G=G, T=400, B=200, H=100, r=100, S=8, d=d, dtype=dtype, seed=31 + G, kv4=True)


def test_gqa_one_head_per_unit_is_the_one_head_handle():
    # groups = 1 is the ordinary handle: identical outputs, victims, state
    U, T, B, H, r, S, d = 4, 300, 100, 50, 50, 6, 128
    Q, K, V, q, k, v = _rand(9, U, 1, T, S, d, "bf16")
    scale = 1.0 / np.sqrt(d)
    a = Dev("h2o", U, d, B, H, r, "bf16", scale)
    b = Dev("h2o", U, d, B, H, r, "bf16", scale, groups=1)
    a.prefill(Q, K, V)
    b.prefill(Q, K, V)
    for t in range(S):
        oa, va = a.step(q[t], k[t], v[t])
        ob, vb = b.step(q[t], k[t], v[t])
        assert (oa == ob).all() and (va == vb).all()
    sa, sb = a.state(), b.state()
    for key in ("K", "V", "score", "pos", "occ", "npos"):
        assert (sa[key] == sb[key]).all(), key
    a.close()
    b.close()


def test_gqa_prefill_statistics():
    U, G, T, d = 3, 4, 257, 128
    Q, K, V, *_ = _rand(31, U, G, T, 0, d, "bf16", key_scale=2.0)
    scale = 1.0 / np.sqrt(d)
    dev = Dev("h2o", U, d, 64, 32, 32, "bf16", scale, groups=G)
    dev.prefill(Q, K, V)
    m, l, c = dev.stats(T)
    mo, lo, co = oracle.prefill_scores(Q, np.repeat(K, G, axis=0), scale)
    np.testing.assert_allclose(m, mo, rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(l, lo, rtol=1e-4)
    _, cu, _, _, _ = oracle.h2o_prefill_gqa(Q, K, V, 64, 32, 32, scale)
    check_scores(c, cu, "unit column sums")
    # each query row distributes probability 1: a unit's prompt mass is G * T
    np.testing.assert_allclose(c.sum(axis=1), G * T, rtol=1e-5)
    dev.close()


def test_gqa_workload_units():
    # the grouped-query benchmark workload's inputs on a subset of its units
    w = wl.WORKLOADS["gqa-8x8x4"]
    units = list(range(6))
    g = wl.generate(w, units=units, steps=16)
    dev = Dev("h2o", len(units), w.head_dim, w.budget, w.heavy, w.recent, w.dtype, w.scale, groups=w.groups)
    dev.prefill(g["Q"], g["K"], g["V"])
    s = dev.state()
    st, _, near0 = align_prefill(s, g["Q"], g["K"], g["V"], w.budget, w.heavy, w.recent, w.scale)
    assert (s["pos"] == st.pos).all() and rows_equal(s, st)
    check_scores(s["score"], st.score, "prompt scores")
    near, _ = h2o_lockstep(dev, st, g["q"], g["k"], g["v"], w.prompt, w.recent, w.scale, check_every=4)
    record("gqa-8x8x4 lockstep", near_ties=near0 + near)
    dev.close()


def test_gqa_rejects_bad_groups():
    s = torch.cuda.current_stream()
    for groups, budget in ((0, 64), (17, 64), (4, 1025)):
        with pytest.raises(L.H2OError):
            L.h2o_init_gqa(budget, budget // 2, budget - budget // 2, 1, 2, groups, 128, L.H2O_BF16, 0.1, s)
    # the cluster of a grouped-query cache is its query heads: no split to set
    h = L.h2o_init_gqa(64, 32, 32, 1, 2, 4, 128, L.H2O_BF16, 0.1, s)
    with pytest.raises(L.H2OError) as e:
        L.h2o_set_decode_split(h, 2)
    assert e.value.code == L.H2O_ERR_STATE
    L.h2o_destroy(h)
