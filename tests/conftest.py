import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU")
    config.addinivalue_line("markers", "slow: full-size workload")


def pytest_collection_modifyitems(config, items):
    """Skip GPU tests cleanly when no CUDA device is present (they are deselected
    with ``-m "not gpu"`` anyway)."""
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


# Values the tests give the planner overrides, as text (parametrised cases),
# and the override field values they stand for (None: the planner's choice).
_KNOB_VALUES = {
    "tile_n": lambda v: int(v),
    "cta_pair": lambda v: int(v),                             # "0": no pairs, "1": pairs
    "tail_split": lambda v: 1 if str(v) == "force" else int(v),   # "force": split short tiles too
    "tail_halves": lambda v: -1 if str(v) == "1" else int(v),     # "0": off
    "cluster_split": lambda v: -1 if str(v) == "1" else int(v),   # "0": through the workspace
    "seg_first": lambda v: int(v),                            # "0": segments last, "1": first
}


@pytest.fixture
def knobs():
    """Sets planner overrides for one test (accumulating over calls):
    ``knobs(tile_n="128")``; ``knobs(tile_n=None)`` returns that one to the
    planner. Every override is cleared when the test ends."""
    import dense_gemm_persistent_gb300 as dg
    state = {}

    def setk(**kw):
        for name, v in kw.items():
            if v is None:
                state.pop(name, None)
            else:
                state[name] = _KNOB_VALUES[name](v) if name in _KNOB_VALUES else int(v)
        dg.set_overrides(**state)

    yield setk
    dg.set_overrides()
