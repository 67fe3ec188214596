import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def pytest_collection_modifyitems(config, items):
    # GPU tests cannot run without a device; skip rather than fail on CPU hosts
    # when someone selects them explicitly.
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


def pytest_terminal_summary(terminalreporter):
    """How much of the AdamW tolerance the GPU parity checks used, per test:
    the largest error relative to the oracle's result of master, exp_avg and
    exp_avg_sq, the elements beyond a strict 1e-6 of the result, and the bf16
    parameters' distance in ulps from the oracle's."""
    try:
        from tests.helpers import MARGINS
    except Exception:  # pragma: no cover
        return
    if not MARGINS:
        return
    per = {}
    for rec in MARGINS:
        agg = per.setdefault(rec["case"], {})
        kind = rec["kind"]
        agg[kind + "_n"] = agg.get(kind + "_n", 0) + rec["n"]
        for k, v in rec.items():
            if k.startswith("max_"):
                agg[k] = max(agg.get(k, 0), v)
            elif k.startswith("n_"):
                agg[k] = agg.get(k, 0) + v
    tr = terminalreporter
    tr.section("AdamW parity margins (GPU vs oracle)")
    tr.write_line("case | state elems | max rel err master / exp_avg / exp_avg_sq | "
                  "beyond 1e-6 of result master / exp_avg / exp_avg_sq | bf16 elems | "
                  "max ulp | at 1 ulp | beyond 1 ulp")
    for case, a in per.items():
        tr.write_line(
            f"{case} | {a.get('state_n', 0)} | "
            f"{a.get('max_rel_master', 0):.2e} / {a.get('max_rel_exp_avg', 0):.2e} / "
            f"{a.get('max_rel_exp_avg_sq', 0):.2e} | "
            f"{a.get('n_beyond_1e-6_master', 0)} / {a.get('n_beyond_1e-6_exp_avg', 0)} / "
            f"{a.get('n_beyond_1e-6_exp_avg_sq', 0)} | {a.get('bf16_n', 0)} | "
            f"{a.get('max_ulp', 0)} | {a.get('n_off_by_1_ulp', 0)} | {a.get('n_beyond_1_ulp', 0)}")
