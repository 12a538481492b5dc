"""The README's decode-step example runs as written and its result matches
the fp64 oracle (write the step's rows at the manager's slots, then attend)."""
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
pytestmark = pytest.mark.gpu


def test_readme_decode_example():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    text = open(os.path.join(ROOT, "README.md")).read()
    code = re.search(r"```python\n(.*?)```", text, re.S).group(1)
    env = {}
    exec(compile(code, "README.md", "exec"), env)
    import oracle.paged_ops as ops
    k, v = env["k_cache"].cpu(), env["v_cache"].cpu()
    # the pools after the call hold the new rows at the manager's slots
    kr, vr = torch.zeros_like(k), torch.zeros_like(v)
    ops.write_kv(kr, vr, env["key"].cpu(), env["value"].cpu(), env["slots"].tolist())
    assert torch.equal(k, kr) and torch.equal(v, vr)
    ref = ops.attend(env["q"].cpu(), kr, vr, env["tables"], env["lens"].cpu().tolist(),
                     env["D"] ** -0.5)
    err = (env["out"].cpu().double() - ref).abs().max().item()
    assert err <= 2e-3, err
