import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(scope="session")
def cuda_lib():
    """The CUDA path's binding; a GPU test fails loudly if it cannot load."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("gpu test run without a CUDA device")
    import paged_kv_gqa_write_gb300 as pa
    pa.load()
    return pa


def pytest_terminal_summary(terminalreporter):
    """The largest |GPU - oracle| of every comparison the parity helpers made
    (FP32 outputs against the 5e-3 gate; BF16 outputs as a fraction of their
    per-element bound), worst first per test file."""
    try:
        from pa_testutil import ERRORS
    except ImportError:
        return
    if not ERRORS:
        return
    import json
    log = os.environ.get("PA_MAXERR_LOG")
    if log:
        with open(log, "w") as f:
            json.dump([{"test": t, "what": w, "max_err": m, "bound": b} for t, w, m, b in ERRORS],
                      f, indent=1)
    tr = terminalreporter
    tr.section("max |err| against the oracle (worst per test)")
    worst = {}
    for t, w, m, b in ERRORS:
        if t not in worst or m / b > worst[t][1] / worst[t][2]:
            worst[t] = (w, m, b)
    for t in sorted(worst, key=lambda k: -worst[k][1] / worst[k][2]):
        w, m, b = worst[t]
        tr.write_line(f"{m:10.3e} / {b:.1e}  {t}  [{w}]")
