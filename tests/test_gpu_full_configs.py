"""Parity at the full sizes of every workload, in the launch configuration
the benchmark uses (all units in one handle, automatic split).  The oracle
replays sampled units one by one; every unit is checked against invariants
that hold at any size."""
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

from parity import run_full_config   # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,sample", [
    ("tiny", [0, 1, 2, 3]),
    ("opt-6.7b", [0, 131, 255]),
    ("hashevict-opt-6.7b", [0, 131, 255]),
    ("opt-30b", [0, 1791, 3583]),
    ("llama-7b-32k", [7]),
])
def test_full_size_workload(name, sample):
    near = run_full_config(name, sample)
    print("%s: near ties forced %d" % (name, near))


@pytest.mark.parametrize("name,sample", [
    ("gqa-8x8x4", [0, 37, 63]),
])
def test_full_size_grouped_query(name, sample):
    near = run_full_config(name, sample)
    print("%s: near ties forced %d" % (name, near))


@pytest.mark.parametrize("name,sample", [
    ("opt-6.7b", [0, 131, 255]),
    ("opt-30b", [0, 1791, 3583]),
])
def test_full_size_persistence_rule(name, sample):
    flips = run_full_config(name, sample, rule="sh")
    print("%s persistence rule: flag flips %d" % (name, flips))
