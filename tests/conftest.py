import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built det_gemm library")
    config.addinivalue_line("markers", "slow: large inputs; minutes rather than seconds")


def pytest_collection_modifyitems(config, items):
    # GPU tests without a GPU are skipped here rather than failed, so that
    # `-m "not gpu"` and a bare run both work on a CPU-only machine. With a
    # GPU present they run, and a missing library fails them loudly.
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    # Parity rates of the BF16 comparisons against the oracle (see
    # tests/gpu_util.py, RATES): printed, and written as JSON lines to the
    # file DET_GEMM_RATES_OUT names, if any.
    mod = sys.modules.get("gpu_util")
    rates = getattr(mod, "RATES", None) if mod is not None else None
    if not rates:
        return
    tr = terminalreporter
    tr.write_sep("-", "BF16 parity rates against the oracle")
    tr.write_line("%-44s %9s %9s %9s %9s %8s" % ("comparison", "elements", "bit-eq", "<=1ulp(S)", "<=1ulp(C)", "max/ulpS"))
    for what, n, same, s1, lit, worst in rates:
        tr.write_line("%-44s %9d %9.5f %9.5f %9.5f %8.3f" % (what[:44], n, same, s1, lit, worst))
    out = os.environ.get("DET_GEMM_RATES_OUT")
    if out:
        import json
        with open(out, "w") as f:
            for what, n, same, s1, lit, worst in rates:
                f.write(json.dumps({"what": what, "elements": n, "bit_equal": same, "within_1ulp_S": s1,
                                    "within_1ulp_C": lit, "max_diff_ulp_S": worst}) + "\n")
