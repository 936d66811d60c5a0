"""The usage example in README.md runs as printed and computes what its
comments say (slots 53 and 149; the gathered rows 37 and 43 are the new
tokens' keys)."""
import os
import re

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_readme_python_example():
    text = open(os.path.join(ROOT, "README.md")).read()
    block = re.search(r"```python\n(.*?)```", text, flags=re.S).group(1)
    env = {}
    exec(compile(block, "README.md", "exec"), env)
    assert env["slots"].cpu().tolist() == [53, 149]
    k_out, key = env["k_out"], env["key"]
    assert torch.equal(k_out[37].view(torch.int16), key[0, 0].view(torch.int16))
    assert torch.equal(k_out[43].view(torch.int16), key[0, 1].view(torch.int16))
    assert int(env["err"].item()) == 0
