"""The README's usage example runs as written (and its outputs have the documented shapes)."""

import os

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_readme_python_example_runs():
    import torch
    from differential_attention_03_gb300 import build
    build.build()
    text = open(os.path.join(ROOT, "README.md")).read()
    start = text.index("```python") + len("```python")
    code = text[start:text.index("```", start)]
    env = {}
    exec(compile(code, "README.md", "exec"), env)
    torch.cuda.synchronize()
    from differential_attention_03_gb300 import binding as da
    da.device_status()
    B, n, H, d = env["B"], env["n"], env["H"], env["d"]
    assert env["y"].shape == (B, n, H, 2 * d) and bool(torch.isfinite(env["y"].float()).all())
    assert env["out"].shape == (B, H, 2 * d) and bool(torch.isfinite(env["out"].float()).all())
    assert env["grads"]["dq1"].shape == (B, n, H, 64) and bool(torch.isfinite(env["grads"]["dv"]).all())
