"""The usage example of the README runs as written (forward, residual output,
backward, optional terms, status check)."""
import re
from pathlib import Path

import pytest

pytestmark = pytest.mark.gpu


def test_readme_usage_example_runs():
    text = (Path(__file__).resolve().parents[1] / "README.md").read_text()
    blocks = re.findall(r"```python\n(.*?)```", text, re.S)
    assert blocks, "no python block in the README"
    env = {}
    exec(compile(blocks[0], "README.md", "exec"), env)
    import torch
    torch.cuda.synchronize()
    for name in ("o", "lse", "o_lo", "dq", "dk", "dv", "o2", "lse2"):
        assert name in env, name
        assert bool(torch.isfinite(env[name].float()).all()), name
