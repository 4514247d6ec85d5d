"""Eviction ties on the device.

The eviction rule breaks score ties to the lowest slot [H2O review page,
提案手法: greedy eviction of the token with the least accumulated attention;
the tie rule is the reading this library takes].  These cases make the tie
exact on both sides: every cached key of a unit equals the new key, so every
attention row is uniform and every live slot gains the very same
probability in fp32 and in fp64; states loaded with duplicated scores then
tie exactly among several candidates, which sit in shuffled slots.  The
device's victims must equal the oracle's bit for bit, with no near-tie
allowance, on one CTA per unit and on a cluster of four (the cross-CTA
arg-min), and for a cache shared by four query heads.

The hand-worked trajectory of tests/golden/h2o_equal_keys.json (prompt of
four identical keys, budget three) runs through the prompt phase and three
decode steps with its victims, positions and scores in twelfths.
"""
import json
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

import oracle                                     # noqa: E402
from kv_cache_eviction_h2o_gb300 import binding as L   # noqa: E402
from kv_cache_eviction_h2o_gb300 import workloads as wl   # noqa: E402
from parity import Dev, check_out, check_scores, record   # noqa: E402

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


def _bf16_bits(x):
    return (np.ascontiguousarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)


@pytest.mark.parametrize("split,groups", [(1, 0), (4, 0), (0, 4)])
def test_exact_ties_take_the_lowest_slot(split, groups):
    U, d, B, H, r, S = 6, 128, 410, 205, 205, 24
    G = max(groups, 1)
    scale = 1.0 / np.sqrt(d)
    rng = np.random.default_rng(31 + split + groups)
    bf = lambda *s: wl.round_bf16(rng.standard_normal(s, dtype=np.float32))
    key = bf(U, d)                                  # one key per unit, shared by every slot
    K = np.repeat(key[:, None, :], B, axis=1)
    V = bf(U, B, d)
    score = rng.integers(0, 3, size=(U, B)).astype(np.float64) * 0.25   # three exact values
    pos = np.stack([rng.permutation(B) for _ in range(U)]).astype(np.int32)
    occ = np.full(U, B, np.int32)
    npos = np.full(U, B, np.int32)
    dev = Dev("h2o", U, d, B, H, r, "bf16", scale, split=split, groups=groups)
    try:
        L.h2o_set_state(dev.h, _bf16_bits(K), _bf16_bits(V), score, pos, None, occ, npos)
        st = oracle.H2OState(U, B, d)
        st.K[:] = K; st.V[:] = V; st.score[:] = score; st.pos[:] = pos; st.occ[:] = occ
        step = oracle.h2o_decode_step_gqa if G > 1 else oracle.h2o_decode_step
        ties = 0
        for t in range(S):
            p = B + t
            q = bf(U * G, d)
            v = bf(U, d)
            out_g, vic_g = dev.step(q, key, v)
            out_o, vic_o, mg, _ = step(st, q, key, v, p, r, scale)
            ties += int((mg == 0).sum())
            assert (vic_g == vic_o).all(), "step %d: victims %s, the lowest tied slots %s" % (
                t, vic_g.tolist(), vic_o.tolist())
            check_out(out_g, out_o, "step %d out" % t)
            g = dev.state()
            assert (g["pos"] == st.pos).all(), "step %d: positions differ" % t
            check_scores(g["score"], st.score, "step %d scores" % t)
        # the case really is a tie at (nearly) every decision
        assert ties >= S * U // 2, ties
        record("ties split=%d groups=%d" % (split, groups), exact_ties=ties, decisions=S * U)
    finally:
        dev.close()


@pytest.mark.parametrize("split", [1, 2])
def test_hand_worked_equal_keys_trajectory(split):
    with open(os.path.join(HERE, "golden", "h2o_equal_keys.json")) as f:
        g = json.load(f)
    T, B, H, r = g["T"], g["B"], g["H"], g["r"]
    d, scale = 64, 0.125
    rng = np.random.default_rng(41)
    key = rng.standard_normal(d, dtype=np.float32)
    Q = rng.standard_normal((1, T, d), dtype=np.float32)
    K = np.tile(key, (1, T, 1))
    V = rng.standard_normal((1, T, d), dtype=np.float32)
    dev = Dev("h2o", 1, d, B, H, r, "f32", scale, split=split)
    try:
        dev.prefill(Q, K, V)
        s0 = dev.state()
        assert s0["pos"][0].tolist() == g["prefill_pos"]
        np.testing.assert_allclose(s0["score"][0] * 12, g["prefill_score_12ths"], atol=1e-6 * 12)
        vals = {j: V[0, j].astype(np.float64) for j in range(T)}
        pos = list(g["prefill_pos"])
        for s in g["steps"]:
            qn = rng.standard_normal((1, d), dtype=np.float32)
            vn = rng.standard_normal((1, d), dtype=np.float32)
            cached = [vals[p] for p in pos]
            out, vic = dev.step(qn, key[None, :], vn)
            assert int(vic[0]) == s["victim"]
            st = dev.state()
            assert st["pos"][0].tolist() == s["pos"]
            np.testing.assert_allclose(st["score"][0] * 12, s["score_12ths"], atol=1e-6 * 12)
            check_out(out, ((sum(cached) + vn[0]) / 4)[None, :], "p=%d out" % s["p"])
            pos = s["pos"]
            vals[s["p"]] = vn[0].astype(np.float64)
    finally:
        dev.close()
