"""The repository's front-page usage example (its first python block) runs as
written: forward, residual output, backward, optional terms, status check."""
import re
from pathlib import Path

import pytest

pytestmark = pytest.mark.gpu


def test_readme_usage_example_runs():
    text = (Path(__file__).resolve().parents[1] / "README.md").read_text()
    blocks = re.findall(r"```python\n(.*?)```", text, re.S)
    assert blocks, "no python block on the front page"
    env = {}
    exec(compile(blocks[0], "usage-example", "exec"), env)
    import torch
    torch.cuda.synchronize()
    for name in ("o", "lse", "o_lo", "dq", "dk", "dv", "o2", "lse2"):
        assert name in env, name
        assert bool(torch.isfinite(env[name].float()).all()), name
