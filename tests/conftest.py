import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# Achieved errors of the parity tests, per case and tensor (printed at the end of the session and,
# when PARITY_MARGINS_OUT names a file, written there as JSON).
_MARGINS = {}


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


@pytest.fixture(scope="session")
def cuda_lib():
    """The built C-ABI library (skips when no GPU is present)."""
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from softmax_attention_chunk_gb300 import path_attn

    return path_attn


@pytest.fixture(scope="session")
def record_margin():
    """record_margin(case, tensor, max_abs_err, bound, max_abs_ref=None, rel_fro=None)."""

    def rec(case, name, err, bound, ref_max=None, rel=None):
        entry = {"max_abs_err": float(err), "bound": float(bound)}
        if ref_max is not None:
            entry["max_abs_ref"] = float(ref_max)
        if rel is not None:
            entry["rel_fro"] = float(rel)
        _MARGINS.setdefault(case, {})[name] = entry

    return rec


def pytest_sessionfinish(session, exitstatus):
    if not _MARGINS:
        return
    out = os.environ.get("PARITY_MARGINS_OUT")
    if out:
        with open(out, "w") as f:
            json.dump(_MARGINS, f, indent=1, sort_keys=True)
    lines = ["parity margins (max abs err / bound):"]
    for case in sorted(_MARGINS):
        parts = [f"{n} {v['max_abs_err']:.2e}/{v['bound']:.1e}" for n, v in sorted(_MARGINS[case].items())]
        lines.append(f"  {case}: " + ", ".join(parts))
    print("\n" + "\n".join(lines))
