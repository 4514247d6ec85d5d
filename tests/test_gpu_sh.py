"""The persistence-of-importance cache (sh_init) on the GPU against the
oracle (Scissorhands abstract: tokens that were pivotal keep mattering; the
rule read from it: pivotal = probability above the uniform share of the
tokens attended, a 32-step history per slot, evict the fewest pivotal
steps, then the oldest).  Histories, positions, victims and cache rows are
compared bit-exactly; a flag may differ only where the oracle's P * m is
within 1e-4 of 1 at that decision (counted, and the oracle then follows the
device); outputs within the usual tolerance."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

import oracle                                              # noqa: E402
from kv_cache_eviction_h2o_gb300 import binding as L       # noqa: E402
from kv_cache_eviction_h2o_gb300 import workloads as wl    # noqa: E402
from parity import record, Dev, rows_equal, sh_align_prefill, sh_lockstep  # noqa: E402

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


def _run(U, T, B, H, r, S, d, dtype, seed, split=0, key_scale=1.5, inputs=None):
    Q, K, V, q, k, v = inputs if inputs is not None else _rand(seed, U, T, S, d, dtype, key_scale)
    scale = 1.0 / np.sqrt(d)
    dev = Dev("sh", U, d, B, H, r, dtype, scale, split=split)
    dev.prefill(Q, K, V)
    s = dev.state()
    st, f0 = sh_align_prefill(s, Q, K, V, B, H, r, scale)
    assert (s["pos"] == st.pos).all(), "prompt positions differ"
    assert (s["code"] == st.mask).all(), "prompt histories differ"
    assert rows_equal(s, st), "prompt cache rows differ"
    f1, st = sh_lockstep(dev, st, q, k, v, T, r, scale)
    dev.close()
    return f0, f1


@pytest.mark.parametrize("T,B,H,r", [
    (5, 8, 4, 4),            # append phase
    (1, 8, 4, 4),            # single-token prompt (its one row decides nothing)
    (31, 20, 10, 10),        # prompt shorter than the history window
    (32, 20, 10, 10),
    (33, 20, 10, 10),        # the first row falls out of the window
    (40, 8, 0, 8),           # no candidates from the prompt: sliding window
    (40, 8, 8, 0),           # no recent window
    (40, 1, 1, 0),           # one slot
    (70, 33, 17, 16),        # ragged stages
    (300, 200, 100, 100),    # several stages per warp
    (1500, 1100, 600, 500),  # budget above one CTA's chunk: a cluster splits it
])
@pytest.mark.parametrize("dtype,d", [("f32", 64), ("bf16", 128)])
def test_sh_edge_cases(T, B, H, r, dtype, d):
    _run(U=3, T=T, B=B, H=H, r=r, S=40, d=d, dtype=dtype, seed=13 * T + B)


@pytest.mark.parametrize("split", [1, 3, 16])
def test_sh_opt67b_units(split):
    # the OPT-6.7B-shaped workload's inputs on 12 units, past the 32-step
    # history (a flag set in the prompt's last row leaves it at step 32)
    w = wl.WORKLOADS["opt-6.7b"]
    g = wl.generate(w, units=list(range(12)), steps=40)
    f0, f1 = _run(U=12, T=w.prompt, B=w.budget, H=w.heavy, r=w.recent, S=40, d=w.head_dim, dtype=w.dtype,
                  seed=0, split=split, inputs=(g["Q"], g["K"], g["V"], g["q"], g["k"], g["v"]))
    record("persistence rule opt-6.7b split=%d" % split, flips=f0 + f1)


def test_sh_one_cta_with_a_budget_near_the_chunk_limit():
    _run(U=2, T=1300, B=1000, H=500, r=500, S=6, d=128, dtype="bf16", seed=78, split=1)


def test_sh_zero_logits_keep_a_sliding_window():
    # queries orthogonal to every key: every probability is the uniform
    # share, nothing is pivotal, the cache is always the newest B tokens
    U, T, B, H, r, S, d = 4, 100, 40, 20, 20, 20, 128
    g = np.random.default_rng(5)
    Q = np.zeros((U, T, d), np.float32); K = np.zeros((U, T, d), np.float32)
    q = np.zeros((S, U, d), np.float32); k = np.zeros((S, U, d), np.float32)
    Q[..., :64] = wl.round_bf16(g.standard_normal((U, T, 64), dtype=np.float32))
    K[..., 64:] = wl.round_bf16(g.standard_normal((U, T, 64), dtype=np.float32))
    q[..., :64] = wl.round_bf16(g.standard_normal((S, U, 64), dtype=np.float32))
    k[..., 64:] = wl.round_bf16(g.standard_normal((S, U, 64), dtype=np.float32))
    V = wl.round_bf16(g.standard_normal((U, T, d), dtype=np.float32))
    v = wl.round_bf16(g.standard_normal((S, U, d), dtype=np.float32))
    dev = Dev("sh", U, d, B, H, r, "bf16", 1.0 / np.sqrt(d))
    dev.prefill(Q, K, V)
    s = dev.state()
    assert (s["code"] == 0).all() and (np.sort(s["pos"], axis=1) == np.arange(T - B, T)).all()
    for t in range(S):
        dev.step(q[t], k[t], v[t])
        s = dev.state()
        assert (s["code"] == 0).all()
        assert (np.sort(s["pos"], axis=1) == np.arange(T + t + 1 - B, T + t + 1)).all()
    dev.close()


def test_sh_wrong_calls_are_refused():
    s = torch.cuda.current_stream()
    with pytest.raises(L.H2OError):
        L.sh_init(64, 32, 32, 1, 2, 128, L.H2O_BF16 | L.H2O_KV8, 0.1, s)
    h = L.sh_init(64, 32, 32, 1, 2, 128, L.H2O_BF16, 0.1, s)
    x = torch.zeros((2, 16, 128), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((2, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(L.H2OError):
        L.h2o_prefill(h, x, x, x, 16)               # an H2O call on this handle
    with pytest.raises(L.H2OError):
        L.sh_decode_step(h, y, y, y, torch.empty((2, 128), device="cuda"))   # before a prompt
    L.h2o_destroy(h)
