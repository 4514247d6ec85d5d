"""The allocation-free prompt scorer.

Callers that cannot allocate device memory -- serving runtimes that reserve
all device memory for their own pool at start-up, hosts whose allocation
calls may synchronise the device in the middle of their own work -- use
h2o_prompt_scores_noalloc, whose scratch is a fixed array inside the
library.  Its column sums must match those of the regular entry point,
h2o_prefill, and the CPU oracle's, on consecutive calls that reuse that
array: the tensor-core path (bf16, head_dim 128), the CUDA-core path (fp32,
head_dim 64), and a call that fills the array exactly.

This file is collected last so that a failure here stops a ``-x`` run only
after every other test has run.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

import oracle   # noqa: E402

pytestmark = pytest.mark.gpu

SCORE_RTOL, SCORE_ATOL = 1e-4, 1e-12     # the accumulated-score tolerance of the parity tests


def _lib():
    import __graft_entry__
    __graft_entry__.build()
    from kv_cache_eviction_h2o_gb300 import binding as L
    return L


def _inputs(seed, U, T, d, dtype):
    g = torch.Generator().manual_seed(seed)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    Q = torch.randn(U, T, d, generator=g).to(tdt).cuda()
    K = (2.0 * torch.randn(U, T, d, generator=g)).to(tdt).cuda()
    V = torch.randn(U, T, d, generator=g).to(tdt).cuda()
    return Q, K, V


def _regular(L, Q, K, V, batch, heads, T, d, cdt, scale):
    h = L.h2o_init(16, 8, 8, batch, heads, d, cdt, scale, torch.cuda.current_stream())
    try:
        L.h2o_prefill(h, Q, K, V, T)
        c = np.empty((batch * heads, T))
        L.h2o_get_prefill_stats(h, None, None, c)
    finally:
        L.h2o_destroy(h)
    return c


def _close(got, want, what):
    bad = np.abs(got - want) > SCORE_RTOL * np.abs(want) + SCORE_ATOL
    assert not bad.any(), "%s: %d column sums differ (worst %g)" % (what, bad.sum(), np.abs(got - want).max())


def _noalloc(L, Q, K, batch, heads, T, d, cdt, scale):
    c_dev = torch.full((batch * heads, T), float("nan"), dtype=torch.float64, device="cuda")
    L.h2o_prompt_scores_noalloc(Q, K, batch, heads, T, d, cdt, scale, c_dev, torch.cuda.current_stream())
    torch.cuda.synchronize()
    got = c_dev.cpu().numpy()
    assert np.isfinite(got).all(), "column sums left unwritten or a wait ran out (NaN)"
    return got


@pytest.mark.parametrize("dtype,d,cases", [
    # two calls in a row on the shared scratch, the second with other sizes
    ("bf16", 128, ((1, 2, 4, 300), (2, 1, 3, 1000))),
    ("f32", 64, ((3, 1, 2, 77), (4, 2, 1, 513))),
])
def test_noalloc_scores_match_prefill_and_oracle_on_consecutive_calls(dtype, d, cases):
    L = _lib()
    cdt = L.H2O_BF16 if dtype == "bf16" else L.H2O_F32
    scale = 1.0 / np.sqrt(d)
    for seed, batch, heads, T in cases:
        Q, K, V = _inputs(seed, batch * heads, T, d, dtype)
        got = _noalloc(L, Q, K, batch, heads, T, d, cdt, scale)
        _close(got, _regular(L, Q, K, V, batch, heads, T, d, cdt, scale), "seed %d vs h2o_prefill" % seed)
        _, _, c_ref = oracle.prefill_scores(Q.float().cpu().numpy(), K.float().cpu().numpy(), scale)
        _close(got, c_ref, "seed %d vs the oracle" % seed)


def test_noalloc_at_its_maximum_size():
    # batch * heads * T equal to the array's capacity: the normaliser half of
    # the scratch ends exactly at the array's end
    L = _lib()
    d, batch, heads = 128, 1, 256
    T = L.H2O_NOALLOC_MAX_TOKENS // (batch * heads)
    scale = 1.0 / np.sqrt(d)
    Q, K, V = _inputs(5, batch * heads, T, d, "bf16")
    got = _noalloc(L, Q, K, batch, heads, T, d, L.H2O_BF16, scale)
    _close(got, _regular(L, Q, K, V, batch, heads, T, d, L.H2O_BF16, scale), "max size vs h2o_prefill")
    # two units against the oracle, and the column sums of every unit add up to T
    for u in (0, batch * heads - 1):
        _, _, c_ref = oracle.prefill_scores(Q[u:u + 1].float().cpu().numpy(), K[u:u + 1].float().cpu().numpy(), scale)
        _close(got[u:u + 1], c_ref, "max size unit %d vs the oracle" % u)
    np.testing.assert_allclose(got.sum(axis=1), T, rtol=1e-5)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    L = _lib()
    d = 64
    T = L.H2O_NOALLOC_MAX_TOKENS // 2 + 1
    Q = torch.zeros((16,), dtype=torch.float32, device="cuda")
    c = torch.zeros((16,), dtype=torch.float64, device="cuda")
    with pytest.raises(L.H2OError) as e:
        # the raw call: the binding's own size checks would stop the tiny buffers first
        rc = L.lib().h2o_prompt_scores_noalloc(Q.data_ptr(), Q.data_ptr(), 1, 2, T, d, L.H2O_F32, 0.125,
                                               c.data_ptr(), torch.cuda.current_stream().cuda_stream)
        L._check(rc)
    assert e.value.code == L.H2O_ERR_ARG
    assert "exceeds" in str(e.value)
