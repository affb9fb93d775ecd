import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: large parity cases")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def cuda_device():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test collected on a machine without a CUDA device")
    return torch.device("cuda", 0)


@pytest.fixture(scope="session")
def pkv_lib():
    """Build (if stale) and load libpagedkv.so; no GPU needed to load it."""
    from paged_kv_cache_102_gb300 import build as pkv_build
    pkv_build.build()
    import paged_kv_cache_102_gb300 as pkv
    pkv.load()
    return pkv


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Print every attention parity comparison's largest error as a fraction
    of the plain tolerance (over the elements held to it) and of each
    element's bound, and write them as JSON when PKV_PARITY_REPORT names a
    file."""
    try:
        from tests.parity import RESULTS
    except Exception:
        return
    if not RESULTS:
        return
    worst = max(RESULTS, key=lambda r: r[3])
    tr = terminalreporter
    tr.write_sep("-", f"attention parity: {len(RESULTS)} comparisons; largest max|err|/tol over elements held "
                      f"to the plain tol = {worst[3]:.3f} ({worst[0]}); largest max|err|/bound = "
                      f"{max(r[4] for r in RESULTS):.3f}")
    for name, err, tol, frac_plain, frac_bound, n, n_extra in sorted(RESULTS, key=lambda r: -r[3])[:12]:
        tr.write_line(f"  plain {frac_plain:6.3f}  bound {frac_bound:6.3f}  max|err| {err:.3e}  tol {tol:.0e}  "
                      f"elements {n:>8}  half-ulp allowed {n_extra:>5}  {name}")
    path = os.environ.get("PKV_PARITY_REPORT")
    if path:
        with open(path, "w") as f:
            json.dump([dict(test=r[0], max_err=r[1], tol=r[2], max_err_over_tol_plain_elements=r[3],
                            max_err_over_bound=r[4], elements=r[5], half_ulp_elements=r[6]) for r in RESULTS],
                      f, indent=1)
