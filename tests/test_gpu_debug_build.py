"""GPU: the parity suites re-run against the CPATTN_DEBUG build of the library.

compute-sanitizer is closed on this machine.  In its place, libcpattn_debug.so is
built from the same sources with CPATTN_DEBUG defined: the tensor-core kernels
then check every tensor row they compute (TMA tile rows, statistics loads,
epilogue stores) against that tensor's extent, and a failed check latches
CPATTN_ERR_BOUNDS in the device status word and skips the access.  Every parity
test calls cpattn_check, so one failed check anywhere fails the run; the
results must still match the oracle."""
import os
import subprocess
import sys

import pytest

from conftest import ROOT

pytestmark = pytest.mark.gpu

SUITES = ["tests/test_gpu_ring.py", "tests/test_gpu_partial.py", "tests/test_gpu_partial_bwd.py",
          "tests/test_gpu_allgather.py", "tests/test_gpu_packed.py", "tests/test_gpu_canary.py",
          "tests/test_gpu_ulysses.py"]


def test_parity_suites_pass_under_bounds_checks():
    import __graft_entry__
    __graft_entry__._build_lib().build(debug=True)
    env = dict(os.environ, CPATTN_DEBUG_LIB="1")
    probe = subprocess.run(
        [sys.executable, "-c", "import blockwise_online_softmax_cpattn_gb300 as cp; "
         "print(cp.LIB_PATH)"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert probe.returncode == 0, probe.stderr[-2000:]
    assert probe.stdout.strip().endswith("libcpattn_debug.so"), probe.stdout
    r = subprocess.run([sys.executable, "-m", "pytest", *SUITES, "-m", "gpu", "-x", "-q",
                        "-p", "no:cacheprovider"], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
