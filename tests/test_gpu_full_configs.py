"""Parity at the full sizes of every workload, in the launch configuration
the benchmark uses (all units in one handle, automatic split).  The oracle
replays sampled units one by one (at least 16 per workload, 4 of the
32-unit long-context layer, whose 32768-token prompt is the oracle's
longest job); every unit is checked against invariants that hold at any
size.  Near ties (H2O decisions where the oracle's candidate scores lie
within 1e-6 of each other) and flag flips are counted and recorded."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

from parity import record, run_full_config   # noqa: E402
from kv_cache_eviction_h2o_gb300 import workloads as wl   # noqa: E402

pytestmark = pytest.mark.gpu


def sample(name, n):
    """n units spread over the workload (first and last included), seeded."""
    U = wl.WORKLOADS[name].units
    if n >= U:
        return list(range(U))
    rest = np.random.default_rng(len(name) * 7 + n).choice(np.arange(1, U - 1), n - 2, replace=False)
    return sorted({0, U - 1, *rest.tolist()})


@pytest.mark.parametrize("name,n", [
    ("tiny", 4),
    ("opt-6.7b", 16),
    ("hashevict-opt-6.7b", 16),
    ("opt-30b", 16),
    ("llama-7b-32k", 4),
])
def test_full_size_workload(name, n):
    units = sample(name, n)
    near = run_full_config(name, units)
    record("full %s" % name, near_ties=near, sampled_units=len(units))


def test_full_size_grouped_query():
    units = sample("gqa-8x8x4", 16)
    near = run_full_config("gqa-8x8x4", units)
    record("full gqa-8x8x4", near_ties=near, sampled_units=len(units))


@pytest.mark.parametrize("name,n", [
    ("opt-6.7b", 16),
    ("opt-30b", 16),
])
def test_full_size_persistence_rule(name, n):
    units = sample(name, n)
    flips = run_full_config(name, units, rule="sh")
    record("full %s persistence rule" % name, flips=flips, sampled_units=len(units))
