import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU oracle test")


def pytest_collection_modifyitems(config, items):
    # GPU tests skip cleanly when no GPU is present, so `-m "not gpu"` and a
    # plain run on a CPU machine both pass.
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA GPU")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Print the achieved parity errors of this run (margins to the
    tolerances) after the test results."""
    try:
        from _harness import RECORDS
    except Exception:  # pragma: no cover
        return
    if not RECORDS:
        return
    tr = terminalreporter
    tr.section("parity errors achieved")
    fwd = [(w, r) for w, r in RECORDS if "o_max_abs" in r]
    for w, r in fwd:
        tr.write_line(f"{w}: O max-abs {r['o_max_abs']:.2e} (over 1e-2: {r['o_flat_over']}/"
                      f"{r['o_n']}, storage-bound use {r['o_bound_use']:.2f}) rel-fro "
                      f"{r['o_rel_fro']:.2e}, LSE {r['lse_max_abs']:.1e}")
    for w, r in RECORDS:
        g = {k: v for k, v in r.items() if k in ("dq", "dc", "dw", "dgamma")}
        if g:
            tr.write_line(f"{w}: gradients rel-fro " + ", ".join(f"{k} {v:.2e}" for k, v in g.items()))
    for w, r in RECORDS:
        if "block" in r:
            tr.write_line(f"{w}: rel-fro " + ", ".join(f"{k} {v:.2e}" for k, v in r["block"].items()))
    grads = {}
    for w, r in RECORDS:
        for k, v in r.items():
            if k in ("dq", "dc", "dw", "dgamma") and v > grads.get(k, (0.0, ""))[0]:
                grads[k] = (v, w)
    if fwd:
        w, r = max(fwd, key=lambda x: x[1]["o_max_abs"])
        over = sum(r["o_flat_over"] for _, r in fwd)
        n = sum(r["o_n"] for _, r in fwd)
        tr.write_line(f"WORST O max-abs {r['o_max_abs']:.3e} at {w} (b,s,h)={r['o_worst_bsh']}, "
                      f"storage error there {r['o_storage_at_worst']:.2e}; flat 1e-2 "
                      f"{'met' if over == 0 else f'NOT met by {over} of {n} elements'}; "
                      f"worst O rel-fro {max(x['o_rel_fro'] for _, x in fwd):.2e} (<= 5e-3)")
    if grads:
        tr.write_line("WORST gradient rel-fro (<= 1e-2): " + ", ".join(
            f"{k} {v:.2e} ({w})" for k, (v, w) in grads.items()))
