"""bench.py's launch contract, checked on the CPU: --gpus N without N ranks is refused."""

import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("impl", ["ours", "reference"])
def test_gpus_without_ranks_is_refused(impl):
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--steps", "1",
                        "--warmup", "3", "--impl", impl], capture_output=True, text=True, env=env, timeout=120)
    assert r.returncode != 0
    assert "n_gpus" not in r.stdout
    assert "WORLD_SIZE" in r.stderr
