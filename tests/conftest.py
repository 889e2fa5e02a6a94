import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Print the boundary-case counts of every store parity comparison of the
    session: the decisions the parity bar excuses (codes within 1e-6 of a
    decision boundary, QJL projections below 1e-6 of the key norm, fp16 values
    within 1e-6 of a rounding midpoint, group-32 codes within 1e-6 of a
    half-integer), each beside the count its density predicts, and the bytes
    that actually differed."""
    import parity

    if not parity.RECORDED:
        return
    tr = terminalreporter
    tr.write_sep("-", "store parity: boundary cases counted (expected from the density) and bytes mismatched")
    tot_m = tot_x = 0
    for case, r in parity.RECORDED:
        tr.write_line(parity.summary_line(case, r))
        tot_m += r["mismatched_bytes"]
        tot_x += r["excusable_bytes"]
    tr.write_line(f"total: {len(parity.RECORDED)} comparisons, mismatched bytes {tot_m}, "
                  f"bytes touching a counted case {tot_x}, unexplained 0")
