"""The warp-per-unit H2O decode kernel (thousands of one-head units: every
warp owns whole units, w, w + W, ...) against the oracle.

From eight units per SM on (1216 on 152 SMs) each warp streams whole units;
the counts below put one or two units on every warp, with a ragged last
round, and the warps' stage rings run from one unit into the next.  Positions, occupancy and (quantised) cache rows are
compared bit-exactly, victims up to counted near ties, outputs and scores
within the usual tolerances (H2O decode rule: accumulate each slot's
probability, evict the lowest score outside the recent window, lowest slot
on ties)."""
import numpy as np
import pytest

import oracle
from kv_cache_eviction_h2o_gb300 import workloads as wl
from parity import Dev, align_prefill, check_scores, h2o_lockstep, record, rows_equal

pytestmark = pytest.mark.gpu


def _draw(rng, dtype, *shape):
    x = rng.standard_normal(shape).astype(np.float32)
    return wl.round_bf16(x) if dtype == "bf16" else x


def _run(U, T, B, H, r, S, d, dtype, bits, seed, key_scale=1.0, check_every=2):
    rng = np.random.default_rng(seed)
    Q, V = _draw(rng, dtype, U, T, d), _draw(rng, dtype, U, T, d)
    K = _draw(rng, dtype, U, T, d) * np.float32(key_scale)
    q, v = _draw(rng, dtype, S, U, d), _draw(rng, dtype, S, U, d)
    k = _draw(rng, dtype, S, U, d) * np.float32(key_scale)
    if dtype == "bf16":
        K, k = wl.round_bf16(K), wl.round_bf16(k)
    scale = 1.0 / np.sqrt(d)
    dev = Dev("h2o", U, d, B, H, r, dtype, scale, kv8=bits == 8, kv4=bits == 4)
    dev.prefill(Q, K, V)
    s = dev.state()
    st, _, near0 = align_prefill(s, Q, K, V, B, H, r, scale)
    if bits:
        st = oracle.kv8(st, bits)
    assert (s["pos"] == st.pos).all()
    assert rows_equal(s, st)
    check_scores(s["score"], st.score, "prompt scores")
    near, _ = h2o_lockstep(dev, st, q, k, v, T, r, scale, check_every=check_every)
    dev.close()
    return near0 + near


@pytest.mark.parametrize("bits", [0, 8, 4])
@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64), ("f32", 128), ("bf16", 64)])
def test_warp_kernel_matches_oracle(dtype, d, bits):
    # 2500 units: one or two per warp; budget 60 = four stages, the last ragged
    near = _run(U=2500, T=90, B=60, H=30, r=30, S=6, d=d, dtype=dtype, bits=bits, seed=101 + d + bits)
    record("warp units %s d%d q%d" % (dtype, d, bits), near_ties=near)


@pytest.mark.parametrize("bits", [0, 4])
def test_warp_kernel_opt67b_rows(bits):
    # the OPT-6.7B budget (410 slots: 26 stages per unit) on 1300 units
    w = wl.WORKLOADS["opt-6.7b"]
    near = _run(U=1300, T=450, B=w.budget, H=w.heavy, r=w.recent, S=4, d=128, dtype="bf16", bits=bits,
                seed=7 + bits, check_every=3)
    record("warp units opt-6.7b budget q%d" % bits, near_ties=near)


@pytest.mark.parametrize("T,B,H,r", [
    (5, 8, 4, 4),            # append phase: the cache fills during the steps
    (40, 8, 0, 8),           # sliding window
    (40, 8, 8, 0),           # no recent window
    (40, 1, 1, 0),           # one slot
    (1030, 1024, 512, 512),  # the largest budget the kernel takes
])
@pytest.mark.parametrize("bits", [0, 4])
def test_warp_kernel_edge_cases(T, B, H, r, bits):
    near = _run(U=1300, T=T, B=B, H=H, r=r, S=8 if B < 1024 else 3, d=64 if B == 1024 else 128, dtype="bf16",
                bits=bits, seed=3 * T + B + bits, check_every=4)
    record("warp units edge T%d B%d q%d" % (T, B, bits), near_ties=near)
