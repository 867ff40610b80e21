import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def cuda_device():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def pytest_terminal_summary(terminalreporter):
    """Attention error figures of the GPU parity tests: one line per full-size
    workload, and the worst case over every other comparison by output dtype.
    With PAGEDKV_ERROR_STATS=<path> they are also written there as JSON."""
    helpers = sys.modules.get("gpu_helpers")
    stats = getattr(helpers, "ERROR_STATS", None) if helpers else None
    if not stats:
        return
    tr = terminalreporter
    tr.section("attention error vs the fp64 oracle (max-abs, max-rel over max(|o|, 1e-3))")
    rest = {}
    for what, dt, n, ma, mr in stats:
        if what.startswith("full-size"):
            tr.write_line(f"{what:<34} {dt:<9} {n:>10} elements  max-abs {ma:.3e}  max-rel {mr:.3e}")
        else:
            c, a, r = rest.get(dt, (0, 0.0, 0.0))
            rest[dt] = (c + 1, max(a, ma), max(r, mr))
    for dt, (c, a, r) in sorted(rest.items()):
        tr.write_line(f"{'all other comparisons (' + str(c) + ')':<34} {dt:<9} {'':>10}           "
                      f"max-abs {a:.3e}  max-rel {r:.3e}")
    path = os.environ.get("PAGEDKV_ERROR_STATS")
    if path:
        import json
        with open(path, "w") as f:
            json.dump([list(x) for x in stats], f)
