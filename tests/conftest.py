import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Parity maxima of every GPU-vs-oracle comparison of the run (max|dO|, max|dLSE|,
    max|O_ref|, the O bound applied).  FA_PARITY_REPORT=<path> also writes them as JSON."""
    pu = sys.modules.get("parity_util")
    if pu is None or not pu.RECORDS:
        return
    tr = terminalreporter
    tr.section("parity maxima (GPU vs fp64 oracle)")
    for what, dtype, d_o, d_lse, max_o, bound, rows in pu.RECORDS:
        tr.write_line(f"{what[:70]:70s} {dtype:5s} rows {rows:>9d}  max|dO| {d_o:.3e}  "
                      f"max|dLSE| {d_lse:.3e}  max|O_ref| {max_o:7.3f}  bound {bound}")
    path = os.environ.get("FA_PARITY_REPORT")
    if path:
        keys = ("what", "dtype", "max_abs_dO", "max_abs_dLSE", "max_abs_O_ref", "O_bound", "rows")
        with open(path, "w") as f:
            json.dump([dict(zip(keys, r)) for r in pu.RECORDS], f, indent=1)
