"""Failure detection on the GPU without faulting it: a bounded wait that runs
out is reported by h2o_sync and leaves the handle usable; host-side fault
injection makes allocations and launches fail cleanly."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

from kv_cache_eviction_h2o_gb300 import binding as L   # noqa: E402
from parity import Dev  # noqa: E402

pytestmark = pytest.mark.gpu


def _small():
    g = np.random.default_rng(1)
    U, T, d = 2, 40, 64
    Q = g.standard_normal((U, T, d), dtype=np.float32)
    K = g.standard_normal((U, T, d), dtype=np.float32)
    V = g.standard_normal((U, T, d), dtype=np.float32)
    q = g.standard_normal((U, d), dtype=np.float32)
    return Q, K, V, q


def test_bounded_wait_timeout_is_reported_and_recoverable():
    Q, K, V, q = _small()
    dev = Dev("h2o", 2, 64, 8, 4, 4, "f32", 0.125)
    dev.prefill(Q, K, V)
    L.h2o_selftest_wait_timeout(dev.h)
    with pytest.raises(L.H2OError) as e:
        L.h2o_sync(dev.h)
    assert e.value.code == L.H2O_ERR_DEVICE_TIMEOUT
    # the error word was cleared and the context still works
    L.h2o_sync(dev.h)
    out, vic = dev.step(q, q, q)
    assert np.isfinite(out).all()
    dev.close()


def test_injected_allocation_failure(monkeypatch):
    monkeypatch.setenv("H2O_FAULT", "alloc")
    with pytest.raises(L.H2OError) as e:
        L.h2o_init(8, 4, 4, 1, 2, 64, L.H2O_F32, 0.125, torch.cuda.current_stream())
    assert e.value.code == L.H2O_ERR_ALLOC
    monkeypatch.delenv("H2O_FAULT")
    h = L.h2o_init(8, 4, 4, 1, 2, 64, L.H2O_F32, 0.125, torch.cuda.current_stream())
    L.h2o_destroy(h)


def test_injected_launch_failure(monkeypatch):
    Q, K, V, q = _small()
    dev = Dev("h2o", 2, 64, 8, 4, 4, "f32", 0.125)
    dev.prefill(Q, K, V)
    qd = torch.from_numpy(q).cuda()
    monkeypatch.setenv("H2O_FAULT", "launch")
    with pytest.raises(L.H2OError) as e:
        L.h2o_decode_step(dev.h, qd, qd, qd, dev.out, dev.victim)
    assert e.value.code == L.H2O_ERR_CUDA
    monkeypatch.delenv("H2O_FAULT")
    out, vic = dev.step(q, q, q)
    assert np.isfinite(out).all()
    dev.close()
