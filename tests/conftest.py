import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def pytest_sessionfinish(session, exitstatus):
    """With AWQ_BOUNDS_REPORT set (a run against the bounds-checked library), write the library's record of
    failed bounds checks to that file when the session ends."""
    path = os.environ.get("AWQ_BOUNDS_REPORT")
    if not path:
        return
    from post_bit_weight_awq_b300 import capi_testing

    failures, unit, line, offset = capi_testing.awq_bounds_report()
    with open(path, "w") as f:
        f.write(f"{failures} {unit} {line} {offset}\n")
