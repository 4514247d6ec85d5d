"""Per-head cache policies on the device against the oracle.

["Model Tells You What to Discard" review page, method section: every head
is profiled on the prompt and takes the first of its cache policies whose
recovery of the head's attention reaches a threshold; Figure 2 caption: the
"Frequency + Local" policy is the H2O cache.]  The workloads mix local,
heavy-hitter and broad heads so that every policy is taken.

Checked against the oracle (oracle.fg_profile / fg_prefill /
fg_decode_step):
* each unit's policy, bit-exact -- one may differ only where the recovery
  that decides it lies within 1e-4 of the threshold (fp32 sums on the
  device, fp64 in the oracle); such flips are counted and the oracle then
  follows the device's choice;
* both recoveries within 1e-4;
* the kept prompt positions and their scores (as h2o_prefill's);
* every decode step: victims (near ties as for h2o_decode_step), outputs,
  positions and scores, each unit with its own budget and window, all in
  one launch.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

import oracle   # noqa: E402
from kv_cache_eviction_h2o_gb300 import workloads as wl   # noqa: E402
from parity import Dev, accept_victims, check_out, check_scores, kept_lists, record   # noqa: E402

pytestmark = pytest.mark.gpu
REC_TOL = 1e-4


def _profile_and_align(dev, g, w, tau, Bf):
    """Device policies and caches against the oracle's; returns the oracle's
    per-unit states and parameters (following the device where a policy
    sits within REC_TOL of the threshold) and the number of such flips."""
    U = w.units if g["Q"].shape[0] == w.units else g["Q"].shape[0]
    pol_o, rl_o, rf_o = oracle.fg_profile(g["Q"], g["K"], w.budget, w.heavy, w.recent, w.scale, tau)
    pol_g, rl_g, rf_g = dev.policy()
    assert np.abs(rl_g - rl_o).max() <= REC_TOL, np.abs(rl_g - rl_o).max()
    assert np.abs(rf_g - rf_o).max() <= REC_TOL, np.abs(rf_g - rf_o).max()
    flips = 0
    for u in np.nonzero(pol_g != pol_o)[0]:
        near = abs(rl_o[u] - tau) < REC_TOL or abs(rf_o[u] - tau) < REC_TOL
        assert near, "unit %d: policy %d, oracle %d (recoveries %r %r)" % (u, pol_g[u], pol_o[u], rl_o[u], rf_o[u])
        flips += 1
    states, params = [], []
    near = 0
    st_dev = dev.state()
    T = g["Q"].shape[1]
    for u in range(U):
        Bu, Hu, ru = oracle.fg_policy_params(pol_g[u], w.budget, w.heavy, w.recent, Bf)
        st, c, kept, margin = oracle.h2o_prefill(g["Q"][u:u + 1], g["K"][u:u + 1], g["V"][u:u + 1], Bu, Hu, ru,
                                                 w.scale)
        kg = kept_lists(st_dev["pos"][u:u + 1], dev.B)[0][:Bu]
        if not (kg == kept[0]).all():
            assert margin[0] < 1e-6, "unit %d: kept positions differ (margin %g)" % (u, margin[0])
            near += 1
            st = oracle.build_cache(g["K"][u:u + 1], g["V"][u:u + 1], c, kg[None], Bu)
        assert (st_dev["pos"][u, :Bu] == st.pos[0]).all(), "unit %d: slot positions differ" % u
        assert (st_dev["pos"][u, Bu:] == -1).all(), "unit %d: slots past its budget in use" % u
        check_scores(st_dev["score"][u, :Bu], st.score[0], "unit %d prompt scores" % u)
        states.append(st)
        params.append((Bu, Hu, ru))
    return pol_g, states, params, flips, near


def _lockstep(dev, states, params, g, T, scale):
    near = 0
    U = len(states)
    for t in range(g["q"].shape[0]):
        p = T + t
        out_g, vic_g = dev.step(g["q"][t], g["k"][t], g["v"][t])
        st_dev = dev.state()
        for u in range(U):
            st, out_o, nt = accept_victims(oracle.h2o_decode_step, states[u], g["q"][t][u:u + 1],
                                           g["k"][t][u:u + 1], g["v"][t][u:u + 1], p, params[u][2], scale,
                                           vic_g[u:u + 1])
            states[u] = st
            near += nt
            Bu = params[u][0]
            check_out(out_g[u:u + 1], out_o, "step %d unit %d out" % (t, u))
            assert (st_dev["pos"][u, :Bu] == st.pos[0]).all(), "step %d unit %d: positions differ" % (t, u)
            assert st_dev["occ"][u] == st.occ[0] and st_dev["npos"][u] == p + 1
            check_scores(st_dev["score"][u, :Bu], st.score[0], "step %d unit %d scores" % (t, u))
            assert (st_dev["K"][u, :Bu] == st.K[0]).all(), "step %d unit %d: cache rows differ" % (t, u)
    return near


@pytest.mark.parametrize("name,units,steps", [
    ("fastgen-tiny", None, None),
    ("fastgen-opt-6.7b", [0, 1, 2, 3, 4, 5, 33, 64], 24),
])
def test_per_head_policies_match_the_oracle(name, units, steps):
    w = wl.WORKLOADS[name]
    g = wl.generate(w, units=units, steps=steps)
    U = g["Q"].shape[0]
    T = w.prompt
    dev = Dev("fg", U, w.head_dim, w.budget, w.heavy, w.recent, w.dtype, w.scale, fg=(w.full_budget, w.tau))
    try:
        dev.prefill(g["Q"], g["K"], g["V"])
        pol, states, params, flips, near0 = _profile_and_align(dev, g, w, w.tau, w.full_budget)
        assert set(pol.tolist()) == {0, 1, 2}, pol          # the mix exercises every policy
        near = _lockstep(dev, states, params, g, T, w.scale)
        record("fastgen %s" % name, policy_flips=flips, near_ties=near0 + near, units=U)
    finally:
        dev.close()


@pytest.mark.parametrize("T", [40, 64])
def test_prompt_within_budget_takes_the_local_policy(T):
    # T <= budget: both recoveries are 1 and every head keeps its whole prompt
    w = wl.WORKLOADS["fastgen-tiny"]
    g = wl.generate(w, units=range(3), steps=4, prompt=T)
    dev = Dev("fg", 3, w.head_dim, w.budget, w.heavy, w.recent, w.dtype, w.scale, fg=(w.full_budget, w.tau))
    try:
        dev.prefill(g["Q"], g["K"], g["V"])
        pol, rl, rf = dev.policy()
        assert (pol == 0).all()
        np.testing.assert_allclose(rl, 1.0, atol=REC_TOL)
        np.testing.assert_allclose(rf, 1.0, atol=REC_TOL)
        pol_g, states, params, flips, near0 = _profile_and_align(dev, g, w, w.tau, w.full_budget)
        _lockstep(dev, states, params, g, T, w.scale)
    finally:
        dev.close()


def test_policy_profile_on_a_persistent_walk():
    """40 units of the OPT-6.7B-shaped prompt: 640 (unit, block) items, more
    than the resident CTAs, so the band sums of the scorer's second pass are
    taken on CTAs that walk several items."""
    w = wl.WORKLOADS["fastgen-opt-6.7b"]
    g = wl.generate(w, units=list(range(40)), steps=1)
    U = g["Q"].shape[0]
    dev = Dev("fg", U, w.head_dim, w.budget, w.heavy, w.recent, w.dtype, w.scale, fg=(w.full_budget, w.tau))
    try:
        dev.prefill(g["Q"], g["K"], g["V"])
        pol, _, _, flips, near0 = _profile_and_align(dev, g, w, w.tau, w.full_budget)
        record("fastgen persistent walk", policy_flips=flips, near_ties=near0, units=U)
    finally:
        dev.close()


def test_every_head_on_the_full_cache():
    """tau = 1 on diffuse attention (Gaussian queries and keys, a prompt four
    times the budget): no compressed policy recovers the whole attention, so
    every head keeps its full cache and the decode step's launch over the
    compressed policies' units has none."""
    from types import SimpleNamespace
    U, T, S, d = 4, 64, 6, 64
    rng = np.random.default_rng(31)
    f = lambda *shape: rng.standard_normal(shape, dtype=np.float32)
    g = {"Q": f(U, T, d), "K": f(U, T, d), "V": f(U, T, d), "q": f(S, U, d), "k": f(S, U, d), "v": f(S, U, d)}
    w = SimpleNamespace(units=U, budget=16, heavy=8, recent=8, scale=1.0 / np.sqrt(d))
    full = T + S
    dev = Dev("fg", U, d, w.budget, w.heavy, w.recent, "f32", w.scale, fg=(full, 1.0))
    try:
        dev.prefill(g["Q"], g["K"], g["V"])
        pol_g, states, params, flips, near0 = _profile_and_align(dev, g, w, 1.0, full)
        assert (pol_g == 2).all(), pol_g
        _lockstep(dev, states, params, g, T, w.scale)
    finally:
        dev.close()


@pytest.mark.parametrize("split", [1, 2, 4])
def test_per_head_policies_with_a_set_split(split):
    """A decode split set on the handle: both launches (compressed policies,
    full caches) take it, raised where a full cache needs more CTAs."""
    w = wl.WORKLOADS["fastgen-opt-6.7b"]
    g = wl.generate(w, units=[0, 1, 2, 3, 33, 64], steps=8)
    U = g["Q"].shape[0]
    dev = Dev("fg", U, w.head_dim, w.budget, w.heavy, w.recent, w.dtype, w.scale, fg=(w.full_budget, w.tau),
              split=split)
    try:
        dev.prefill(g["Q"], g["K"], g["V"])
        pol, states, params, flips, near0 = _profile_and_align(dev, g, w, w.tau, w.full_budget)
        near = _lockstep(dev, states, params, g, w.prompt, w.scale)
        record("fastgen split=%d" % split, policy_flips=flips, near_ties=near0 + near, units=U)
    finally:
        dev.close()
