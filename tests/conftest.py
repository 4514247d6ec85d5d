import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the CUDA library")
    config.addinivalue_line("markers", "slow: long-running oracle case")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Report the near ties and flag flips the parity tests counted (an H2O
    decision or a pivotal flag where fp32 and fp64 may disagree is counted,
    not failed), on the terminal and in gpurun_out/near_ties.json."""
    parity = sys.modules.get("parity")
    rec = getattr(parity, "RECORD", None)
    if not rec:
        return
    terminalreporter.write_line("near ties / flag flips counted by the parity tests:")
    for name in sorted(rec):
        terminalreporter.write_line("  %s: %s" % (name, json.dumps(rec[name], sort_keys=True)))
    out = os.path.join(ROOT, "gpurun_out")
    try:
        os.makedirs(out, exist_ok=True)
        with open(os.path.join(out, "near_ties.json"), "w") as f:
            json.dump(rec, f, indent=1, sort_keys=True)
    except OSError:
        pass
