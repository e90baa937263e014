import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running oracle case")


def pytest_terminal_summary(terminalreporter):
    """Parity margins of the whole-forward comparisons that ran (worst first), against the bounds
    max|g - o| <= 5e-2 and sum|g - o| / sum|o| <= 1e-2."""
    helpers = sys.modules.get("tests.helpers")
    tr = terminalreporter
    rows = getattr(helpers, "MARGINS", None) if helpers else None
    if rows:
        tr.write_line(f"parity margins ({len(rows)} comparisons; bound max_abs 5e-2, mean_rel 1e-2):")
        for what, ma, mr in rows:
            tr.write_line(f"  {what:<44s} max_abs {ma:.2e} ({ma / 5e-2:5.1%})  mean_rel {mr:.2e} ({mr / 1e-2:5.1%})")
    grows = getattr(helpers, "GRAD_MARGINS", None) if helpers else None
    if grows:
        tr.write_line(f"backward margins ({len(grows)} comparisons; value, bound, value / bound):")
        for what, v, bound in grows:
            tr.write_line(f"  {what:<60s} {v:.3e}  bound {bound:.3e} ({v / bound:5.1%})")
