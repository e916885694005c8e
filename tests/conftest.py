import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libmoe.so")
    config.addinivalue_line("markers", "slow: full-size workload checks")


def pytest_terminal_summary(terminalreporter):
    """The measured parity errors of this session beside their bounds: per
    kind of tensor, the comparison closest to its rel-Frobenius bound and the
    one closest to its max-abs bound, and how many elements exceeded the
    literal 3e-2 (bf16 values above 4, where one bf16 ulp exceeds it)."""
    util = sys.modules.get("tests.gpu_util")
    margins = getattr(util, "MARGINS", None)
    if not margins:
        return
    w = terminalreporter.write_line
    w(f"parity margins: {len(margins)} comparisons")
    for key in sorted({(m["dtype"], m["kind"]) for m in margins}):
        ms = [m for m in margins if (m["dtype"], m["kind"]) == key]
        rf_bound = 5e-3 if key[0] == "bf16" else 1e-5
        worst_rf = max(ms, key=lambda m: m["rel_frob"])
        worst_ma = max(ms, key=lambda m: m["max_abs"] / m["max_abs_bound"])
        over = sum(m["n_over_3e-2"] for m in ms)
        w(f"  {key[0]} {key[1]}: {len(ms)} compared; max rel_frob {worst_rf['rel_frob']:.2e} "
          f"(bound {rf_bound:.0e}, {worst_rf['name']}); max-abs {worst_ma['max_abs']:.2e} of "
          f"bound {worst_ma['max_abs_bound']:.2e} ({worst_ma['name']}, max|ref| "
          f"{worst_ma['max_ref']:.3g}); elements above 3e-2: {over}")
    path = os.environ.get("MOE_PARITY_LOG")
    if path:
        import json
        with open(path, "w") as fh:
            json.dump(margins, fh)
