"""The allocation-free prompt scorer.

Callers that cannot allocate device memory (code running while a stream is
captured into a CUDA graph, serving runtimes that reserve all device memory
at start-up) use h2o_prompt_scores_noalloc, whose scratch is a fixed array
inside the library.  Its column sums must match those of the regular
entry point, h2o_prefill, on consecutive calls that reuse that array.

This file is collected last so that a failure here stops a ``-x`` run only
after every other test has run.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

pytestmark = pytest.mark.gpu

SCORE_RTOL, SCORE_ATOL = 1e-4, 1e-12     # the accumulated-score tolerance of the parity tests


def _inputs(seed, U, T, d):
    g = torch.Generator().manual_seed(seed)
    Q = torch.randn(U, T, d, generator=g).to(torch.bfloat16).cuda()
    K = (2.0 * torch.randn(U, T, d, generator=g)).to(torch.bfloat16).cuda()
    V = torch.randn(U, T, d, generator=g).to(torch.bfloat16).cuda()
    return Q, K, V


def _regular(L, Q, K, V, batch, heads, T, d, scale):
    h = L.h2o_init(16, 8, 8, batch, heads, d, L.H2O_BF16, scale, torch.cuda.current_stream())
    try:
        L.h2o_prefill(h, Q, K, V, T)
        c = np.empty((batch * heads, T))
        L.h2o_get_prefill_stats(h, None, None, c)
    finally:
        L.h2o_destroy(h)
    return c


def test_noalloc_scores_match_prefill_on_consecutive_calls():
    import __graft_entry__
    __graft_entry__.build()
    from kv_cache_eviction_h2o_gb300 import binding as L

    d = 128
    scale = 1.0 / np.sqrt(d)
    stream = torch.cuda.current_stream()
    # two calls in a row on the shared scratch, the second with other sizes
    for seed, batch, heads, T in ((1, 2, 4, 300), (2, 1, 3, 1000)):
        Q, K, V = _inputs(seed, batch * heads, T, d)
        c_dev = torch.full((batch * heads, T), float("nan"), dtype=torch.float64, device="cuda")
        L.h2o_prompt_scores_noalloc(Q, K, batch, heads, T, d, L.H2O_BF16, scale, c_dev, stream)
        torch.cuda.synchronize()
        got = c_dev.cpu().numpy()
        want = _regular(L, Q, K, V, batch, heads, T, d, scale)
        assert np.isfinite(got).all()
        bad = np.abs(got - want) > SCORE_RTOL * np.abs(want) + SCORE_ATOL
        assert not bad.any(), "call (seed %d): %d column sums differ" % (seed, bad.sum())


def test_noalloc_rejects_sizes_beyond_its_scratch():
    from kv_cache_eviction_h2o_gb300 import binding as L
    d = 64
    T = L.H2O_NOALLOC_MAX_TOKENS // 2 + 1
    Q = torch.zeros((16,), dtype=torch.float32, device="cuda")
    c = torch.zeros((16,), dtype=torch.float64, device="cuda")
    with pytest.raises(L.H2OError) as e:
        L.h2o_prompt_scores_noalloc(Q, Q, 1, 2, T, d, L.H2O_F32, 0.125, c, torch.cuda.current_stream())
    assert e.value.code == L.H2O_ERR_ARG
    assert "exceeds" in str(e.value)
