"""The benchmark's reference arm (the CPU oracle) on the host: one JSON line
from rank 0 with the contract's keys, nothing from another rank (as when it
is launched at two ranks), for the default configuration (the OPT-30B-shaped
layer), the long-context configuration (its prompt phase timed on a shorter
prompt and scaled), HashEvict, the grouped-query and
persistence-of-importance legs, and 4-bit cache slots."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ARGS = ["--impl", "reference", "--steps", "1", "--warmup", "0", "--decode-steps", "2", "--oracle-units", "2"]


def _run(extra, rank, world):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + ARGS + extra, env=env, cwd=ROOT,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return [line for line in r.stdout.splitlines() if line.startswith("{")]


@pytest.mark.parametrize("extra", [[], ["--config", "llama-7b-32k"], ["--config", "hashevict-opt-6.7b"],
                                   ["--gqa"], ["--sh"], ["--config", "opt-30b-int4"]])
def test_reference_arm_line(extra):
    lines = _run(extra, 0, 2)
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 1
    for key in ("metric", "value", "unit", "ms_per_step", "higher_is_better", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["metric"].startswith("H2O decode steps/s") and d["unit"] == "steps/s"


def test_reference_arm_other_rank_is_silent():
    assert _run([], 1, 2) == []


def test_bench_byte_model_for_quantised_rows():
    sys.path.insert(0, ROOT)
    import bench
    U, B, d = 10, 300, 128
    full = bench.decode_bytes(U, B, d, 2, False)
    b8 = bench.decode_bytes(U, B, d, 2, False, 8)
    b4 = bench.decode_bytes(U, B, d, 2, False, 4)
    # per slot: two rows of 256, 128 or 64 bytes, the scale pair for codes
    assert (full - b8) == U * (B * (2 * 128 - 8) + (2 * 128 - 8))
    assert (b8 - b4) == U * (B * 2 * 64 + 2 * 64)


def test_bench_prompt_phase_byte_model():
    """The prompt phase's HBM bytes, worked by hand for one unit of four
    tokens, d = 2, budget 2: Q and K (16 + 16 B) read by both passes = 64;
    row max and normaliser written and read = 64; column sums written and
    read = 64; two kept rows of K and V read (16) and two slots written,
    rows of 4 B twice plus position and score pair (2 x 20) = 56."""
    import bench
    assert bench.prefill_bytes(1, 1, 4, 2, 2) == 64 + 64 + 64 + 56
    # grouped queries: two query heads read Q twice as large, keep per-head
    # statistics and column sums, and sum the heads' columns per unit
    assert bench.prefill_bytes(1, 2, 4, 2, 2) == 2 * (32 + 16) + 128 + 128 + 64 + 56
    # budget 8 over four tokens: all four prompt rows read (two more, 16 B),
    # and all eight slots written (six more, 6 x 20 B)
    assert bench.prefill_bytes(1, 1, 4, 2, 8) - bench.prefill_bytes(1, 1, 4, 2, 2) == 16 + 6 * 20


def test_bench_prompt_phase_flop_model():
    """Both score passes take 2 d FLOPs per causal (i, j) pair: one unit of
    two tokens (3 pairs: (0,0), (1,0), (1,1)) at d = 3 is 2 x 2 x 3 x 3 =
    36 FLOPs; the OPT-6.7B-shaped layer (256 units, 2048 tokens, d = 128) is
    275 GFLOP."""
    import bench
    assert bench.prefill_flops(1, 2, 3) == 36
    assert bench.prefill_flops(256, 2048, 128) == 2 * 2 * 256 * 128 * 2048 * 2049 // 2
    assert abs(bench.prefill_flops(256, 2048, 128) / 1e9 - 275.0) < 0.1
