"""The bounds-check build (libdiffattn_bounds.so, -DDIFFATTN_BOUNDS) on the small parity cases.

That build checks every TMA coordinate, tensor-memory address and global store of the kernels
before the access and reports a failed check as DIFFATTN_ERR_BOUNDS.  Here it is built, shown to
catch a checked store out of its limit (a self-test whose store lands inside its own array either
way), and then the small-size parity tests (forward V1 / V2 incl. FP8 QK^T and the host-buffer
pipeline, decode incl. FP8 keys and split states, backward fp32 and bf16 incl. the training pair,
projections and layers: n <= 1100, the host pipeline's token chunks up to n = 9000, and the
persistent d = 128 forward on host item plans of two head groups) run against
it in a child process with DIFFATTN_DEBUG=1: each of them reads the device status after its kernels, so a
failed check fails the test.
"""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SMALL = ("(small_full_compare or test_v1_decode or test_v2_decode or backward_f32 or backward_bf16 "
         "or layer_matches or projection_matches or lambda_outside or zero_tokens or train_pair or host_buffers "
         "or planned_item_groups) and not bench and not long")


def _child_env():
    env = dict(os.environ)
    env["DIFFATTN_DEBUG"] = "1"
    return env


@pytest.fixture(scope="module", autouse=True)
def _built():
    from differential_attention_03_gb300 import build
    build.build(bounds=True)


def test_bounds_build_catches_a_checked_store():
    code = (
        "import torch\n"
        "from differential_attention_03_gb300 import binding as da\n"
        "assert da.bounds_checked(), da.LIB_PATH\n"
        "torch.cuda.init()\n"
        "da.debug_bounds_selftest()\n"
        "try:\n"
        "    da.device_status()\n"
        "except da.DiffAttnError as e:\n"
        "    assert e.status == da.ERR_BOUNDS, e\n"
        "    print('caught', e)\n"
        "else:\n"
        "    raise SystemExit('the out-of-limit store was not reported')\n"
        "assert da.device_status() == da.OK\n"  # cleared, context usable
        "x = torch.ones(4, device='cuda')\n"
        "assert float(x.sum()) == 4.0\n"
    )
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=_child_env(), capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "caught ERR_BOUNDS" in r.stdout


def test_small_parity_cases_pass_under_bounds_checks():
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
           "tests/test_gpu_parity.py", "tests/test_gpu_backward_tc.py", "tests/test_gpu_layer.py",
           "tests/test_gpu_train.py", "-k", SMALL]
    r = subprocess.run(cmd, cwd=ROOT, env=_child_env(), capture_output=True, text=True, timeout=3000)
    tail = (r.stdout + r.stderr)[-4000:]
    assert r.returncode == 0, tail
    assert " passed" in r.stdout and " failed" not in r.stdout, tail
