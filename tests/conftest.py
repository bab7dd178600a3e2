import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_terminal_summary(terminalreporter):
    """Print every GPU parity report (worst relative and absolute score error
    against the oracle, kept blocks, kept-set mismatches excused inside the
    band around p) so that a quiet run records the numbers, not only a pass."""
    mod = sys.modules.get("parity_util")
    reports = getattr(mod, "REPORTS", None) if mod else None
    if not reports:
        return
    terminalreporter.write_line("")
    terminalreporter.write_line("parity reports (GPU vs the fp64 oracle):")
    for r in reports:
        terminalreporter.write_line(
            "  %s: worst_rel %.3g, max_abs %.3g, kept %d/%d blocks, excused %d, kept_tokens %s"
            % (r.get("case", "?"), r["worst_rel"], r["max_abs"], r["kept"], r["blocks"],
               r["excused"], r.get("kept_tokens", "-")))
