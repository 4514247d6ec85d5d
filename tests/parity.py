"""Helpers for the GPU parity tests: drive the CUDA library through its C ABI
(via the ctypes binding) and the CPU oracle on the same seeded inputs, and
compare them with the rules the tests state:

* slot positions, eviction victims, LSH codes: bit-exact;
* an H2O decision may differ only where the device's victim is itself a
  candidate (position <= p - r, or any live slot when there is none) whose
  oracle score lies within 1e-6 (relative) of the smallest candidate score;
  such near-ties are counted (and recorded, see ``record``) and the oracle
  is then forced to the device's choice so both trajectories stay aligned;
* outputs within 2e-3 absolute + 1e-2 relative; accumulated scores within
  1e-4 relative (+1e-12 absolute floor).
"""
import numpy as np
import torch

import oracle
from kv_cache_eviction_h2o_gb300 import binding as L

NEAR_TIE = 1e-6
OUT_ATOL, OUT_RTOL = 2e-3, 1e-2
SCORE_RTOL, SCORE_ATOL = 1e-4, 1e-12

# near ties and flag flips counted by the tests of this pytest run, by test
# name; tests/conftest.py writes them out at the end of the run
RECORD = {}


def record(name, **counts):
    """Add counts (near_ties=..., flips=..., decisions=...) under `name`."""
    r = RECORD.setdefault(name, {})
    for k, v in counts.items():
        r[k] = r.get(k, 0) + int(v)


def tdtype(dtype):
    return torch.bfloat16 if dtype == "bf16" else torch.float32


def cdtype(dtype):
    return L.H2O_BF16 if dtype == "bf16" else L.H2O_F32


def to_dev(x, dtype):
    """float32 numpy holding exactly representable values -> device tensor."""
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to("cuda").to(tdtype(dtype)).contiguous()


def host_elems(dtype, shape):
    return np.empty(shape, np.uint16 if dtype == "bf16" else np.float32)


def widen(a, dtype):
    if dtype == "bf16":
        return (a.astype(np.uint32) << 16).view(np.float32)
    return a


class Dev:
    """One device handle (H2O or LSH) for U units with its own stream;
    groups > 1: an H2O handle whose U cache units are each shared by that
    many query heads (q and out then have U * groups rows)."""

    def __init__(self, kind, U, d, B, H, r, dtype, scale, W=None, split=0, kv8=False, groups=0, fg=None, kv4=False):
        self.kind, self.U, self.d, self.B, self.dtype, self.kv8, self.kv4 = kind, U, d, B, dtype, kv8, kv4
        self.G = max(groups, 1)
        self.stream = torch.cuda.current_stream()
        dt = cdtype(dtype) | (L.H2O_KV8 if kv8 else 0) | (L.H2O_KV4 if kv4 else 0)
        if kind == "fg":
            # fg = (full_budget, tau); the handle holds max(B, full_budget) slots per unit
            self.h = L.fg_init(B, H, r, fg[0], fg[1], 1, U, d, dt, scale, self.stream)
            self.B = max(B, fg[0])
        elif kind == "h2o" and groups:
            self.h = L.h2o_init_gqa(B, H, r, 1, U, groups, d, dt, scale, self.stream)
        elif kind == "sh":
            self.h = L.sh_init(B, H, r, 1, U, d, dt, scale, self.stream)
        elif kind == "h2o":
            self.h = L.h2o_init(B, H, r, 1, U, d, dt, scale, self.stream)
        else:
            self.Wd = torch.from_numpy(np.ascontiguousarray(W, np.float32)).cuda()
            self.h = L.lsh_init(B, r, 1, U, d, dt, scale, self.Wd, self.stream)
        if split:
            L.h2o_set_decode_split(self.h, split)
        self.out = torch.empty((U * self.G, d), dtype=torch.float32, device="cuda")
        self.victim = torch.empty((U,), dtype=torch.int32, device="cuda")

    def prefill(self, Q, K, V):
        self.Qd, self.Kd, self.Vd = (to_dev(x, self.dtype) for x in (Q, K, V))
        T = Q.shape[1]
        if self.kind == "h2o":
            L.h2o_prefill(self.h, self.Qd, self.Kd, self.Vd, T)
        elif self.kind == "fg":
            L.fg_prefill(self.h, self.Qd, self.Kd, self.Vd, T)
        elif self.kind == "sh":
            L.sh_prefill(self.h, self.Qd, self.Kd, self.Vd, T)
        else:
            L.lsh_prefill(self.h, self.Qd, self.Kd, self.Vd, T)
        L.h2o_sync(self.h)

    def step(self, q, k, v):
        qd, kd, vd = (to_dev(x, self.dtype) for x in (q, k, v))
        if self.kind == "h2o":
            L.h2o_decode_step(self.h, qd, kd, vd, self.out, self.victim)
        elif self.kind == "fg":
            L.fg_decode_step(self.h, qd, kd, vd, self.out, self.victim)
        elif self.kind == "sh":
            L.sh_decode_step(self.h, qd, kd, vd, self.out, self.victim)
        else:
            L.lsh_decode_step(self.h, qd, kd, vd, self.out, self.victim)
        L.h2o_sync(self.h)
        return self.out.cpu().numpy().astype(np.float64), self.victim.cpu().numpy()

    def state(self):
        U, B, d = self.U, self.B, self.d
        if self.kv8:
            K = np.empty((U, B, d), np.int8); V = np.empty((U, B, d), np.int8)
        elif self.kv4:
            K = np.empty((U, B, d // 2), np.uint8); V = np.empty((U, B, d // 2), np.uint8)
        else:
            K = host_elems(self.dtype, (U, B, d)); V = host_elems(self.dtype, (U, B, d))
        score = np.empty((U, B)); pos = np.empty((U, B), np.int32)
        code = np.empty((U, B), np.uint32); occ = np.empty(U, np.int32); npos = np.empty(U, np.int32)
        L.h2o_get_state(self.h, K, V, score, pos, code, occ, npos)
        if self.kv8 or self.kv4:
            ks = np.empty((U, B), np.float32); vs = np.empty((U, B), np.float32)
            L.h2o_get_kv_scales(self.h, ks, vs)
            if self.kv4:
                K, V = unpack4(K), unpack4(V)
            return dict(K=K, V=V, ks=ks, vs=vs, score=score, pos=pos, code=code, occ=occ, npos=npos)
        return dict(K=widen(K, self.dtype), V=widen(V, self.dtype), score=score, pos=pos, code=code,
                    occ=occ, npos=npos)

    def policy(self):
        pol = np.empty(self.U, np.int32); rl = np.empty(self.U); rf = np.empty(self.U)
        L.fg_get_policy(self.h, pol, rl, rf)
        return pol, rl, rf

    def stats(self, T):
        m = np.empty((self.U * self.G, T), np.float32); l = np.empty((self.U * self.G, T), np.float32)
        c = np.empty((self.U, T))
        L.h2o_get_prefill_stats(self.h, m, l, c)
        return m, l, c

    def close(self):
        L.h2o_destroy(self.h)


def unpack4(b):
    """Packed 4-bit rows [..., d/2] (offset binary, element 2i in the low
    nibble) -> int8 codes [..., d]."""
    b = b.astype(np.int16)
    out = np.empty(b.shape[:-1] + (2 * b.shape[-1],), np.int8)
    out[..., 0::2] = (b & 0xF) - 8
    out[..., 1::2] = (b >> 4) - 8
    return out


def rows_equal(g, st):
    """Cache rows bit-exact: codes and fp32 scales for a quantised cache
    (int8 or 4-bit), the stored values otherwise."""
    if "ks" in g:
        return ((g["K"] == st.kq).all() and (g["V"] == st.vq).all() and (g["ks"] == st.ks).all()
                and (g["vs"] == st.vs).all())
    return (g["K"] == st.K).all() and (g["V"] == st.V).all()


def check_scores(g, o, what):
    bad = np.abs(g - o) > SCORE_RTOL * np.abs(o) + SCORE_ATOL
    assert not bad.any(), "%s: %d mismatches, worst |d|=%g at %s (dev %r, oracle %r)" % (
        what, bad.sum(), np.abs(g - o).max(), np.argwhere(bad)[0], g[bad][0], o[bad][0])


def check_out(g, o, what):
    bad = np.abs(g - o) > OUT_ATOL + OUT_RTOL * np.abs(o)
    assert not bad.any(), "%s: %d mismatches, worst |d|=%g" % (what, bad.sum(), np.abs(g - o).max())


def kept_lists(pos, B):
    """Ascending kept positions per unit, -1 padded to B."""
    out = np.full((pos.shape[0], B), -1, np.int32)
    for u in range(pos.shape[0]):
        p = np.sort(pos[u][pos[u] >= 0])
        out[u, :len(p)] = p
    return out


def align_prefill(dev_state, Q, K, V, B, H, r, scale):
    """Oracle prompt phase compared with the device's; returns (oracle state,
    oracle column sums, near-tie count).  Fails on any other disagreement.
    Q with more rows than K: a grouped-query cache (Q.shape[0] // K.shape[0]
    heads per unit)."""
    if Q.shape[0] != K.shape[0]:
        st, c, kept_o, margin, _ = oracle.h2o_prefill_gqa(Q, K, V, B, H, r, scale)
    else:
        st, c, kept_o, margin = oracle.h2o_prefill(Q, K, V, B, H, r, scale)
    kept_g = kept_lists(dev_state["pos"], B)
    near = 0
    U, T = c.shape
    for u in range(U):
        if (kept_g[u] == kept_o[u]).all():
            continue
        assert margin[u] < NEAR_TIE, "unit %d: kept set differs with margin %g" % (u, margin[u])
        # the device's choice must be a valid top-H up to the near tie
        go = set(kept_g[u][kept_g[u] >= 0].tolist()); oo = set(kept_o[u][kept_o[u] >= 0].tolist())
        cut = min(c[u][j] for j in oo if j < T - r)
        for j in go ^ oo:
            assert abs(c[u][j] - cut) <= NEAR_TIE * abs(cut) + 1e-300, "unit %d: position %d off the cut" % (u, j)
        near += 1
    if near:
        st = oracle.build_cache(K, V, c, kept_g, B)
    return st, c, near


def accept_victims(step, before, q, k, v, p, r, scale, vic_g):
    """The oracle's step from state `before` (left untouched) against the
    device's victims vic_g.  Where they differ, the device's victim must be
    a live candidate slot (position <= p - r; every live slot when none is)
    whose oracle score after this step's accumulation is within NEAR_TIE
    (relative) of the smallest candidate score; the oracle then follows the
    device.  An append on one side and an eviction on the other always
    fails.  Returns (oracle state after the step, oracle output, number of
    near ties followed)."""
    st = before.copy()
    out_o, vic_o, _, ev_min = step(st, q, k, v, p, r, scale)
    mism = np.nonzero(vic_g != vic_o)[0]
    if len(mism) == 0:
        return st, out_o, 0
    for u in mism:
        n = int(before.occ[u])
        assert vic_o[u] >= 0 and vic_g[u] >= 0, "unit %d: append and eviction disagree (%d vs %d)" % (
            u, vic_g[u], vic_o[u])
        assert 0 <= vic_g[u] < n, "unit %d: victim %d is not a live slot" % (u, vic_g[u])
        cand = before.pos[u, :n] <= p - r
        if not cand.any():
            cand[:] = True
        assert cand[vic_g[u]], "unit %d: victim slot %d (position %d) is inside the recent window" % (
            u, vic_g[u], before.pos[u, vic_g[u]])
    st = before.copy()
    forced = np.full(len(vic_g), -1, np.int32)
    forced[mism] = vic_g[mism]
    out_o, _, _, ev_dev = step(st, q, k, v, p, r, scale, forced)
    for u in mism:
        gap = ev_dev[u] - ev_min[u]
        assert gap <= NEAR_TIE * abs(ev_min[u]) + 1e-300, (
            "unit %d: device victim %d has score %r, the smallest candidate (slot %d) %r: not a near tie" % (
                u, vic_g[u], ev_dev[u], vic_o[u], ev_min[u]))
    return st, out_o, len(mism)


def h2o_lockstep(dev, st, q, k, v, T, r, scale, check_every=1):
    """Run the device and the oracle step by step; returns near-tie count.
    q with more rows than k: a grouped-query cache."""
    near = 0
    S = q.shape[0]
    step = oracle.h2o_decode_step_gqa if q.shape[1] != k.shape[1] else oracle.h2o_decode_step
    for t in range(S):
        p = T + t
        out_g, vic_g = dev.step(q[t], k[t], v[t])
        st, out_o, nt = accept_victims(step, st, q[t], k[t], v[t], p, r, scale, vic_g)
        near += nt
        check_out(out_g, out_o, "step %d out" % t)
        if (t % check_every == 0) or t == S - 1:
            g = dev.state()
            assert (g["pos"] == st.pos).all(), "step %d: positions differ" % t
            assert (g["occ"] == st.occ).all() and (g["npos"] == p + 1).all()
            assert rows_equal(g, st), "step %d: cache rows differ" % t
            check_scores(g["score"], st.score, "step %d scores" % t)
    return near, st


def lsh_lockstep(dev, st, q, k, v, W, T, r, scale, check_every=1):
    S = q.shape[0]
    for t in range(S):
        p = T + t
        out_g, vic_g = dev.step(q[t], k[t], v[t])
        out_o, vic_o = oracle.lsh_decode_step(st, q[t], k[t], v[t], W, p, r, scale)
        assert (vic_g == vic_o).all(), "step %d: LSH victims differ at %s" % (t, np.nonzero(vic_g != vic_o)[0][:8])
        check_out(out_g, out_o, "LSH step %d out" % t)
        if (t % check_every == 0) or t == S - 1:
            g = dev.state()
            assert (g["pos"] == st.pos).all(), "LSH step %d: positions differ" % t
            assert (g["code"] == st.code).all(), "LSH step %d: codes differ" % t
            assert (g["occ"] == st.occ).all()
            assert rows_equal(g, st), "LSH step %d: cache rows differ" % t
    return st


def run_full_config(name, sample, check_every=64, rule=None):
    """The whole workload on the device (every unit, full prompt, every
    decode step, automatic launch configuration as the benchmark uses), with
    the units in `sample` drawn from the seeded numpy recipe and replayed by
    the oracle in lockstep from the device's recorded outputs and victims.
    Every unit is also checked against size-independent invariants.  rule
    "sh": the persistence-of-importance cache on an H2O workload; a
    grouped-query workload (groups > 1) runs a grouped-query H2O handle."""
    from kv_cache_eviction_h2o_gb300 import workloads as wl
    w = wl.WORKLOADS[name]
    kind = "lsh" if w.lsh else ("sh" if rule == "sh" else "h2o")
    U, T, d, B, S, G = w.units, w.prompt, w.head_dim, w.budget, w.steps, w.groups
    g = wl.generate_device(w)
    gs = wl.generate(w, units=sample)
    idx = torch.tensor(sample, device="cuda")
    qidx = torch.tensor([u * G + j for u in sample for j in range(G)], device="cuda")
    g["Q"][qidx] = to_dev(gs["Q"], w.dtype)
    g["q"][:, qidx] = to_dev(gs["q"], w.dtype)
    for key in ("K", "V"):
        g[key][idx] = to_dev(gs[key], w.dtype)
    for key in ("k", "v"):
        g[key][:, idx] = to_dev(gs[key], w.dtype)
    stream = torch.cuda.current_stream()
    dt = cdtype(w.dtype)
    if kind == "lsh":
        W = gs["W"]
        Wd = torch.from_numpy(W).cuda()
        h = L.lsh_init(B, w.recent, w.batch, w.heads, d, dt, w.scale, Wd, stream)
        prefill, step = L.lsh_prefill, L.lsh_decode_step
    elif kind == "sh":
        h = L.sh_init(B, w.heavy, w.recent, w.batch, w.heads, d, dt, w.scale, stream)
        prefill, step = L.sh_prefill, L.sh_decode_step
    elif G > 1:
        h = L.h2o_init_gqa(B, w.heavy, w.recent, w.batch, w.heads, G, d, dt, w.scale, stream)
        prefill, step = L.h2o_prefill, L.h2o_decode_step
    else:
        h = L.h2o_init(B, w.heavy, w.recent, w.batch, w.heads, d, dt, w.scale, stream)
        prefill, step = L.h2o_prefill, L.h2o_decode_step
    prefill(h, g["Q"], g["K"], g["V"], T)
    L.h2o_sync(h)
    st0 = _state_all(h, U, B, d, w.dtype)
    st0 = {k: (v[sample] if getattr(v, "ndim", 0) >= 1 else v) for k, v in st0.items()}
    out = torch.empty((U * G, d), dtype=torch.float32, device="cuda")
    vic = torch.empty((U,), dtype=torch.int32, device="cuda")
    outs, vics, hist = [], [], []
    for t in range(S):
        step(h, g["q"][t], g["k"][t], g["v"][t], out, vic)
        outs.append(out[qidx].cpu().numpy().astype(np.float64))
        vics.append(vic[idx].cpu().numpy())
        if kind == "sh":
            # the sampled units' histories and positions after every step
            pos_t = np.empty((U, B), np.int32); code_t = np.empty((U, B), np.uint32)
            occ_t = np.empty(U, np.int32); np_t = np.empty(U, np.int32)
            L.h2o_get_state(h, None, None, None, pos_t, code_t, occ_t, np_t)
            hist.append(dict(pos=pos_t[sample], code=code_t[sample], occ=occ_t[sample], npos=np_t[sample]))
    L.h2o_sync(h)
    st_all = _state_all(h, U, B, d, w.dtype)
    L.h2o_destroy(h)

    # invariants on every unit: full occupancy, unique positions, the recent
    # window present, next position T + S, finite non-negative scores
    pF = T + S - 1
    assert (st_all["occ"] == min(B, T + S)).all()
    assert (st_all["npos"] == T + S).all()
    pos = st_all["pos"]
    srt = np.sort(pos, axis=1)
    assert (np.diff(srt, axis=1) > 0).all(), "duplicate positions"
    lo = max(0, pF - w.recent + 1)
    if pF - lo + 1 > 0:
        recent = np.arange(lo, pF + 1)
        assert all(np.isin(recent, pos[u]).all() for u in range(U)), "recent window missing"
    if kind == "h2o":
        assert np.isfinite(st_all["score"]).all() and (st_all["score"] >= 0).all()
    if kind == "sh":
        # a slot's history holds no more steps than the token has lived
        age = (T + S - 1) - pos
        nb = np.vectorize(lambda x: bin(int(x)).count("1"))(st_all["code"])
        assert (nb <= np.minimum(32, age + 1)).all(), "history longer than the token's life"

    # the sampled units against the oracle, step by step
    sub = {k: v[sample] if k in ("K", "V", "score", "pos", "code", "occ", "npos") else v for k, v in st_all.items()}
    near = 0
    if kind == "lsh":
        st = oracle.lsh_prefill(gs["Q"], gs["K"], gs["V"], W, B, w.recent)
        replay_lsh(st, gs, W, T, w.recent, w.scale, outs, vics)
        assert (sub["code"] == st.code).all()
    elif kind == "sh":
        st, near = sh_align_prefill(st0, gs["Q"], gs["K"], gs["V"], B, w.heavy, w.recent, w.scale)
        assert (st0["pos"] == st.pos).all(), "prompt positions differ"
        assert (st0["code"] == st.mask).all(), "prompt histories differ"
        n2, st = sh_lockstep(_Recorded(outs, vics, hist), st, gs["q"], gs["k"], gs["v"], T, w.recent, w.scale,
                             check_rows=False)
        near += n2
        assert (sub["code"] == st.mask).all(), "final histories differ"
    else:
        # prompt phase: the device's kept set against the oracle's (near ties counted)
        st, c, near = align_prefill(st0, gs["Q"], gs["K"], gs["V"], B, w.heavy, w.recent, w.scale)
        assert (st0["pos"] == st.pos).all(), "prompt positions differ"
        check_scores(st0["score"], st.score, "prompt scores")
        n2, st = replay_h2o(st, gs, T, w.recent, w.scale, outs, vics)
        near += n2
        check_scores(sub["score"], st.score, "final scores")
    assert (sub["pos"] == st.pos).all(), "final positions differ"
    assert (sub["K"] == st.K).all() and (sub["V"] == st.V).all(), "final cache rows differ"
    return near


class _Recorded:
    """A finished device run played back step by step: its outputs, victims
    and per-step states of the sampled units, in the shape the lockstep
    checkers read from a live handle."""

    def __init__(self, outs, vics, states):
        self.outs, self.vics, self.states, self.t = outs, vics, states, -1

    def step(self, q, k, v):
        self.t += 1
        return self.outs[self.t], self.vics[self.t]

    def state(self):
        return self.states[self.t]


def replay_h2o(st, g, T, r, scale, outs, vics):
    """Replay the oracle's H2O decode steps over the device's recorded
    outputs and victims (near ties counted and followed); returns
    (near-tie count, final oracle state).  q with more rows than k: a
    grouped-query cache."""
    near = 0
    step = oracle.h2o_decode_step_gqa if g["q"].shape[1] != g["k"].shape[1] else oracle.h2o_decode_step
    for t in range(len(outs)):
        st, o_ref, nt = accept_victims(step, st, g["q"][t], g["k"][t], g["v"][t], T + t, r, scale, vics[t])
        near += nt
        check_out(outs[t], o_ref, "step %d out" % t)
    return near, st


def replay_lsh(st, g, W, T, r, scale, outs, vics):
    """Replay the oracle's HashEvict decode steps against the device's
    recorded outputs and victims (victims bit-exact)."""
    for t in range(len(outs)):
        o_ref, v_ref = oracle.lsh_decode_step(st, g["q"][t], g["k"][t], g["v"][t], W, T + t, r, scale)
        assert (vics[t] == v_ref).all(), "step %d: LSH victims differ" % t
        check_out(outs[t], o_ref, "step %d out" % t)
    return st


def _state_all(h, U, B, d, dtype):
    K = host_elems(dtype, (U, B, d)); V = host_elems(dtype, (U, B, d))
    score = np.empty((U, B)); pos = np.empty((U, B), np.int32)
    code = np.empty((U, B), np.uint32); occ = np.empty(U, np.int32); npos = np.empty(U, np.int32)
    L.h2o_get_state(h, K, V, score, pos, code, occ, npos)
    return dict(K=widen(K, dtype), V=widen(V, dtype), score=score, pos=pos, code=code, occ=occ, npos=npos)


# ------------------------------------------------------- persistence of importance
# A pivotal flag is decided in fp32 on the device and in fp64 by the oracle;
# a flag may differ only where the oracle's P * m is within SH_NEAR of 1 at
# that very decision.  Such flips are counted and the oracle then adopts the
# device's histories (and its victim, when the flip changed it), after the
# device's choice is checked to be the rule's choice under its own flags.

SH_NEAR = 1e-4


def _popc(x):
    return bin(int(x)).count("1")


def sh_align_prefill(dev_state, Q, K, V, B, H, r, scale):
    """Oracle prompt phase against the device's; returns (oracle state,
    flips).  Fails on a difference not explained by near-threshold flags."""
    mask, margin, tv = oracle.sh_prompt_masks(Q, K, scale, with_t=True)
    U, T = mask.shape
    kept_o = np.empty((U, B), np.int32)
    for u in range(U):
        oracle.lib().oracle_sh_select(T, B, H, r, np.ascontiguousarray(mask[u]), kept_o[u])
    kept_g = kept_lists(dev_state["pos"], B)
    i0 = max(0, T - 32)
    flips = 0
    mask_g = mask.copy()
    for u in range(U):
        slots = np.argsort(dev_state["pos"][u])[B - (kept_g[u] >= 0).sum():]
        for s in slots:
            j = int(dev_state["pos"][u, s])
            hg, ho = int(dev_state["code"][u, s]), int(mask[u, j])
            if hg == ho:
                continue
            x = hg ^ ho
            for b in range(32):
                if (x >> b) & 1:
                    i = T - 1 - b
                    assert i >= i0 and i >= j, "unit %d token %d: history bit %d outside the window" % (u, j, b)
                    t = tv[u, i - i0, j]
                    assert abs(t - 1.0) < SH_NEAR, "unit %d token %d row %d: flag differs with P*m = %r" % (u, j, i, t)
                    flips += 1
            mask_g[u, j] = hg
        if not (kept_g[u] == kept_o[u]).all():
            # a flip moved a count across the selection cut: every token in
            # the difference must sit within one flag of the cut
            assert (np.abs(tv[u] - 1.0) < SH_NEAR).any(), "unit %d: kept sets differ" % u
            cnt = np.array([_popc(m) for m in mask[u]])
            ko = set(kept_o[u][kept_o[u] >= 0].tolist())
            cut = min(cnt[j] for j in ko if j < T - r)
            for j in ko ^ set(kept_g[u][kept_g[u] >= 0].tolist()):
                assert abs(int(cnt[j]) - int(cut)) <= 1, "unit %d: token %d far from the cut" % (u, j)
            flips += 1
    return oracle.sh_build_cache(K, V, mask_g, kept_g, B), flips


def sh_lockstep(dev, st, q, k, v, T, r, scale, check_every=1, check_rows=True):
    """Device and oracle step by step (histories compared every step);
    returns (flips, final oracle state).  check_rows=False: the device state
    carries no cache rows (compared by the caller)."""
    flips = 0
    B = st.B
    for t in range(q.shape[0]):
        p = T + t
        out_g, vic_g = dev.step(q[t], k[t], v[t])
        before = st.copy()
        out_o, vic_o, _, tv = oracle.sh_decode_step(st, q[t], k[t], v[t], p, r, scale, with_t=True)
        g = dev.state()
        bad = (g["code"] != st.mask).any(axis=1) | (vic_g != vic_o)
        if bad.any():
            forced = np.full(st.U, -1, np.int32)
            for u in np.nonzero(bad)[0]:
                n = int(before.occ[u])
                # this step's flags: bit 0 of every surviving live slot, and
                # the new token's own flag in the slot it took
                fg = {}
                for s in range(n):
                    if s != vic_g[u]:
                        assert (int(g["code"][u, s]) >> 1) == (int(before.mask[u, s]) << 1 & 0xffffffff) >> 1, \
                            "step %d unit %d slot %d: older history bits differ" % (t, u, s)
                        fg[s] = int(g["code"][u, s]) & 1
                newslot = vic_g[u] if vic_g[u] >= 0 else n
                fg[B] = int(g["code"][u, newslot]) & 1
                for s, f in fg.items():
                    want = int(tv[u, s] > 1.0)
                    if f != want:
                        assert abs(tv[u, s] - 1.0) < SH_NEAR, "step %d unit %d slot %d: flag differs with P*m = %r" % (
                            t, u, s, tv[u, s])
                        flips += 1
                # the device's victim must be the rule's choice under its flags
                if n >= B:
                    hist = [((int(before.mask[u, s]) << 1) & 0xffffffff) | fg.get(s, 0) for s in range(n)]
                    hist[vic_g[u]] = ((int(before.mask[u, vic_g[u]]) << 1) & 0xffffffff) | int(tv[u, vic_g[u]] > 1.0)
                    cand = [s for s in range(n) if before.pos[u, s] <= p - r] or list(range(n))
                    best = min(cand, key=lambda s: (_popc(hist[s]), int(before.pos[u, s])))
                    if best != vic_g[u]:
                        # the victim's own flag may be the flipped one
                        hist[vic_g[u]] ^= 1
                        best = min(cand, key=lambda s: (_popc(hist[s]), int(before.pos[u, s])))
                        assert abs(tv[u, vic_g[u]] - 1.0) < SH_NEAR and best == vic_g[u], \
                            "step %d unit %d: device victim %d is not the rule's choice" % (t, u, vic_g[u])
                        flips += 1
                    forced[u] = vic_g[u]
            st = before
            out_o, vic_o, _ = oracle.sh_decode_step(st, q[t], k[t], v[t], p, r, scale, forced)
            st.mask[bad] = g["code"][bad]
        check_out(out_g, out_o, "SH step %d out" % t)
        assert (vic_g == vic_o).all()
        if (t % check_every == 0) or t == q.shape[0] - 1:
            assert (g["pos"] == st.pos).all(), "SH step %d: positions differ" % t
            assert (g["occ"] == st.occ).all() and (g["npos"] == p + 1).all()
            assert (g["code"] == st.mask).all(), "SH step %d: histories differ" % t
            if check_rows:
                assert rows_equal(g, st), "SH step %d: cache rows differ" % t
    return flips, st
