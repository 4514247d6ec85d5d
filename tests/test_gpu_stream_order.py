"""Decode steps of several caches queued back to back on one stream.

No host synchronisation separates the steps, so consecutive decode kernels
overlap through programmatic dependent launch.  A step that follows another
cache's step reads its own cache before its dependency wait; a step that
follows a step of the same cache waits first.  A seeded random interleaving
exercises both, and every output and victim is compared with the oracle
(H2O: Heavy-Hitter Oracle, the decode-phase eviction rule; HashEvict: the
Hamming-distance eviction rule; the grouped-query and persistence-of-importance
caches with the same interleaving)."""
import numpy as np
import pytest
import torch

import oracle
from kv_cache_eviction_h2o_gb300 import binding as L
from kv_cache_eviction_h2o_gb300 import workloads as wl
from parity import (Dev, align_prefill, check_scores, replay_h2o, replay_lsh, rows_equal, to_dev)

pytestmark = pytest.mark.gpu


def _order(counts, seed, repeat_p=0.35):
    """A seeded interleaving of the handles' steps: each entry names the
    handle that advances; a handle repeats with probability repeat_p."""
    rng = np.random.default_rng(seed)
    left = list(counts)
    order, last = [], None
    while sum(left):
        live = [i for i in range(len(left)) if left[i]]
        if last is not None and left[last] and rng.random() < repeat_p:
            i = last
        else:
            i = int(rng.choice(live))
        order.append(i)
        left[i] -= 1
        last = i
    return order


@pytest.mark.parametrize("kv8", [False, True])
def test_interleaved_caches_back_to_back(kv8):
    S = 20
    wa = wl.WORKLOADS["opt-6.7b"]
    wc = wl.WORKLOADS["hashevict-opt-6.7b"]
    ga = wl.generate(wa, units=range(0, 12), steps=S)
    gb = wl.generate(wa, units=range(12, 24), steps=S)
    gc = wl.generate(wc, units=range(0, 10), steps=S)
    W = gc["W"]
    devs = [Dev("h2o", 12, wa.head_dim, wa.budget, wa.heavy, wa.recent, wa.dtype, wa.scale, kv8=kv8),
            Dev("h2o", 12, wa.head_dim, wa.budget, wa.heavy, wa.recent, wa.dtype, wa.scale, kv8=kv8),
            Dev("lsh", 10, wc.head_dim, wc.budget, 0, wc.recent, wc.dtype, wc.scale, W=W, kv8=kv8)]
    gens = [ga, gb, gc]
    for dev, g in zip(devs, gens):
        dev.prefill(g["Q"], g["K"], g["V"])
    st0 = [dev.state() for dev in devs]

    # every step's inputs and outputs live on the device before the first launch
    ins = [{key: to_dev(g[key], dev.dtype) for key in ("q", "k", "v")} for dev, g in zip(devs, gens)]
    outs = [torch.empty((S, dev.U, dev.d), dtype=torch.float32, device="cuda") for dev in devs]
    vics = [torch.empty((S, dev.U), dtype=torch.int32, device="cuda") for dev in devs]
    order = _order([S, S, S], seed=7)
    pairs = list(zip(order[:-1], order[1:]))
    assert any(a == b for a, b in pairs) and any(a != b for a, b in pairs)
    t_of = [0, 0, 0]
    for i in order:
        dev, t = devs[i], t_of[i]
        fn = L.h2o_decode_step if dev.kind == "h2o" else L.lsh_decode_step
        fn(dev.h, ins[i]["q"][t], ins[i]["k"][t], ins[i]["v"][t], outs[i][t], vics[i][t])
        t_of[i] += 1
    torch.cuda.synchronize()
    for dev in devs:
        L.h2o_sync(dev.h)

    T = wa.prompt
    for i, (dev, g) in enumerate(zip(devs, gens)):
        o = [x.astype(np.float64) for x in outs[i].cpu().numpy()]
        v = list(vics[i].cpu().numpy())
        fin = dev.state()
        if dev.kind == "h2o":
            st, _, _ = align_prefill(st0[i], g["Q"], g["K"], g["V"], wa.budget, wa.heavy, wa.recent, wa.scale)
            assert (st0[i]["pos"] == st.pos).all()
            if kv8:
                oracle.kv8(st)
            near, st = replay_h2o(st, g, T, wa.recent, wa.scale, o, v)
            check_scores(fin["score"], st.score, "cache %d final scores" % i)
        else:
            st = oracle.lsh_prefill(g["Q"], g["K"], g["V"], W, wc.budget, wc.recent)
            if kv8:
                oracle.kv8(st)
            replay_lsh(st, g, W, T, wc.recent, wc.scale, o, v)
            assert (fin["code"] == st.code).all()
        assert (fin["pos"] == st.pos).all(), "cache %d: final positions differ" % i
        assert rows_equal(fin, st), "cache %d: final rows differ" % i
        assert (fin["npos"] == T + S).all()
    for dev in devs:
        dev.close()


def test_interleaved_grouped_query_and_persistence_caches():
    # a persistence-of-importance cache, a grouped-query cache and a one-head
    # H2O cache, steps interleaved back to back on one stream
    from parity import SH_NEAR, sh_align_prefill
    S = 20
    wa = wl.WORKLOADS["opt-6.7b"]
    wq = wl.WORKLOADS["gqa-8x8x4"]
    gs = wl.generate(wa, units=range(24, 32), steps=S)
    gq = wl.generate(wq, units=range(0, 6), steps=S)
    ga = wl.generate(wa, units=range(0, 12), steps=S)
    devs = [Dev("sh", 8, wa.head_dim, wa.budget, wa.heavy, wa.recent, wa.dtype, wa.scale),
            Dev("h2o", 6, wq.head_dim, wq.budget, wq.heavy, wq.recent, wq.dtype, wq.scale, groups=wq.groups),
            Dev("h2o", 12, wa.head_dim, wa.budget, wa.heavy, wa.recent, wa.dtype, wa.scale)]
    gens = [gs, gq, ga]
    for dev, g in zip(devs, gens):
        dev.prefill(g["Q"], g["K"], g["V"])
    st0 = [dev.state() for dev in devs]
    ins = [{key: to_dev(g[key], dev.dtype) for key in ("q", "k", "v")} for dev, g in zip(devs, gens)]
    outs = [torch.empty((S, dev.U * dev.G, dev.d), dtype=torch.float32, device="cuda") for dev in devs]
    vics = [torch.empty((S, dev.U), dtype=torch.int32, device="cuda") for dev in devs]
    order = _order([S, S, S], seed=11)
    pairs = list(zip(order[:-1], order[1:]))
    assert any(a == b for a, b in pairs) and any(a != b for a, b in pairs)
    t_of = [0, 0, 0]
    for i in order:
        dev, t = devs[i], t_of[i]
        fn = L.sh_decode_step if dev.kind == "sh" else L.h2o_decode_step
        fn(dev.h, ins[i]["q"][t], ins[i]["k"][t], ins[i]["v"][t], outs[i][t], vics[i][t])
        t_of[i] += 1
    torch.cuda.synchronize()
    for dev in devs:
        L.h2o_sync(dev.h)

    T = wa.prompt
    for i, (dev, g) in enumerate(zip(devs, gens)):
        o = [x.astype(np.float64) for x in outs[i].cpu().numpy()]
        v = list(vics[i].cpu().numpy())
        fin = dev.state()
        if dev.kind == "sh":
            st, _ = sh_align_prefill(st0[i], g["Q"], g["K"], g["V"], wa.budget, wa.heavy, wa.recent, wa.scale)
            loose = np.zeros(dev.U, dtype=bool)
            for t in range(S):
                before = st.copy()
                o_ref, v_ref, mg = oracle.sh_decode_step(st, g["q"][t], g["k"][t], g["v"][t], T + t, wa.recent,
                                                         wa.scale)
                loose |= mg < SH_NEAR
                mism = v[t] != v_ref
                if mism.any():
                    assert (mg[mism] < SH_NEAR).all(), "step %d: victims differ with no flag near the threshold" % t
                    st = before
                    forced = np.where(mism, v[t], -1).astype(np.int32)
                    o_ref, _, _ = oracle.sh_decode_step(st, g["q"][t], g["k"][t], g["v"][t], T + t, wa.recent,
                                                        wa.scale, forced)
                err = np.abs(o[t] - o_ref)
                assert (err <= 2e-3 + 1e-2 * np.abs(o_ref)).all(), "persistence step %d out" % t
            assert (fin["code"][~loose] == st.mask[~loose]).all(), "final histories differ"
        else:
            st, _, _ = align_prefill(st0[i], g["Q"], g["K"], g["V"], dev.B, wa.heavy, wa.recent, wa.scale)
            assert (st0[i]["pos"] == st.pos).all()
            near, st = replay_h2o(st, g, T, wa.recent, wa.scale, o, v)
            check_scores(fin["score"], st.score, "cache %d final scores" % i)
        assert (fin["pos"] == st.pos).all(), "cache %d: final positions differ" % i
        assert rows_equal(fin, st), "cache %d: final rows differ" % i
        assert (fin["npos"] == T + S).all()
    for dev in devs:
        dev.close()
