"""The README's PyTorch example runs as written and its gradients agree with
the explicit forward/backward calls it shows."""
import os
import re

import pytest
import torch

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_readme_example_runs():
    text = open(os.path.join(ROOT, "README.md")).read()
    code = re.search(r"```python\n(.*?)```", text, re.S).group(1)
    env = {}
    exec(compile(code, "README.md", "exec"), env)
    torch.cuda.synchronize()
    x, W, w, ids = env["x"], env["W"], env["w"], env["ids"]
    assert env["y"].shape == (4096, 2048) and env["C"].shape == (256, 2048)
    # autograd's gradients for L = sum(y) equal the explicit backward with dy = 1
    import variable_size_expert_gb300 as mgg
    _, r = mgg.moe_forward(x.detach(), W.detach(), ids, w.detach())
    dx, dW, dw = mgg.moe_backward(torch.ones(4096, 2048, device="cuda"), x.detach(), W.detach(), r, 2)
    torch.cuda.synchronize()
    assert torch.allclose(x.grad.float(), dx, rtol=1e-2, atol=1e-2)
    assert torch.allclose(W.grad.float(), dW, rtol=1e-2, atol=1e-2)
    assert torch.allclose(w.grad, dw, rtol=1e-4, atol=1e-3)
