"""The bounds-checked build (libawq_checked.so): the parity tests of the stages, the layer search, the decode
product and the host-buffer pipeline run against it in a child process and must pass with no failed bounds
check, and the check itself records a planted out-of-range offset without touching memory. This stands in
for a memory checker, which this machine does not offer.
"""
import os
import subprocess
import sys

import pytest
import torch

from post_bit_weight_awq_b300 import build

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SELFTEST = r"""
import torch
from post_bit_weight_awq_b300 import capi, capi_testing
buf = torch.full((64,), 7.0, device="cuda")
assert capi_testing.awq_bounds_report()[0] == 0
capi_testing.awq_bounds_selftest(buf)
failures, unit, line, offset = capi_testing.awq_bounds_report()
assert failures == 1 and unit == 1 and line > 0 and offset == 64, (failures, unit, line, offset)
assert bool(torch.all(buf == 7.0))
assert capi_testing.awq_bounds_report()[0] == 0  # the report clears the record
print("selftest ok")
"""


@pytest.fixture(scope="module")
def checked_lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    build.build()
    return build.build(checked=True)


def _env(lib, report=None):
    env = dict(os.environ, AWQ_LIBRARY=lib)
    if report:
        env["AWQ_BOUNDS_REPORT"] = report
    return env


def test_checked_build_records_a_planted_offset(checked_lib):
    r = subprocess.run([sys.executable, "-c", SELFTEST], cwd=ROOT, env=_env(checked_lib), capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "selftest ok" in r.stdout


def test_parity_suite_under_bounds_checks(checked_lib, tmp_path):
    report = str(tmp_path / "bounds.txt")
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
           "tests/test_gpu_stages.py", "tests/test_gpu_w4a16.py", "tests/test_gpu_pipeline.py",
           "tests/test_gpu_layers.py", "-k", "not full_size"]
    r = subprocess.run(cmd, cwd=ROOT, env=_env(checked_lib, report), capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-4000:]
    failures, unit, line, offset = (int(x) for x in open(report).read().split())
    assert failures == 0, f"{failures} failed bounds checks, first in unit {unit} line {line} offset {offset}"


def test_full_size_layers_under_bounds_checks(checked_lib, tmp_path):
    """The full-size cases (every layer shape the benchmark times, and the
    70B-class decode shapes) under the bounds-checked build: no access
    outside its buffer."""
    report = str(tmp_path / "bounds.txt")
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
           "tests/test_gpu_w4a16.py", "tests/test_gpu_layers.py", "-k", "full_size"]
    r = subprocess.run(cmd, cwd=ROOT, env=_env(checked_lib, report), capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-4000:]
    failures, unit, line, offset = (int(x) for x in open(report).read().split())
    assert failures == 0, f"{failures} failed bounds checks, first in unit {unit} line {line} offset {offset}"
