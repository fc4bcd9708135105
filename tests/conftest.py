import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_terminal_summary(terminalreporter):
    """The largest ulp distance the bf16-criterion checks accepted, per check."""
    mod = sys.modules.get("_util")
    seen = getattr(mod, "ULP_SEEN", None) if mod else None
    if seen:
        terminalreporter.write_line("bf16 criterion: max ulp accepted / fraction within 1 ulp")
        for k in sorted(seen):
            m, f = seen[k]
            terminalreporter.write_line(f"  {k}: {m} ulp, {f:.5f}")
