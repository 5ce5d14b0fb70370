import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Print the error statistics of every oracle comparison made in this session."""
    try:
        import parity
    except ImportError:
        return
    if not parity.RECORDS:
        return
    tr = terminalreporter
    tr.section("parity against the fp64 oracle")
    tr.write_line(f"{'case':<72} {'max|O-O64|':>11} {'lit.region':>11} {'>2e-3':>8} {'elements':>10} {'max|dLSE|':>10}")
    for what, st in parity.RECORDS:
        lse = st.get("lse_max_err")
        tr.write_line(f"{what[:72]:<72} {st['o_max_err_vs_fp64']:>11.3e} {st['o_max_err_vs_fp64_literal_region']:>11.3e} "
                      f"{st['o_over_2e-3']:>8d} {st['o_elements']:>10d} {'-' if lse is None else format(lse, '.3e'):>10}")
