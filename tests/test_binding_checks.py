"""Argument checks of the Python binding, refused before any library call.

ruDNN 0.1.7, src/paged_attention/mod.rs (the torch-facing entry points check
dtype, contiguity, device, shapes against the plan, and refuse an output that
shares storage with an input).  The first group runs on the CPU: the checks
that come before the plan's upload state is consulted.  The second needs an
uploaded plan on the GPU but still launches nothing: every call raises first.
"""
import pytest
import torch

import paged_kv_attention_20_gb300 as pka


def _plan():
    # two sequences (5 and 20 keys, pages of 16), one decode query each
    return pka.paged_attn_plan([5, 20], [[0, 1], [2, 3]], [0, 1], [4, 19], 16, 4, upload=False)


def _tensors(device, dtype=torch.bfloat16):
    q = torch.zeros(2, 4, 64, dtype=dtype, device=device)
    k = torch.zeros(4, 16, 2, 64, dtype=dtype, device=device)
    v = torch.zeros(4, 16, 2, 64, dtype=dtype, device=device)
    return q, k, v


def test_early_refusals_on_the_host(built_lib):
    plan = _plan()
    q, k, v = _tensors("cpu")
    with pytest.raises(TypeError):                                     # dtype outside f32/f16/bf16
        pka.paged_attn_forward(plan, q.to(torch.int32), k, v, 0.125)
    with pytest.raises(TypeError):                                     # caches of another dtype
        pka.paged_attn_forward(plan, q, k.float(), v, 0.125)
    with pytest.raises(ValueError, match="contiguous"):
        pka.paged_attn_forward(plan, q.transpose(0, 1), k, v, 0.125)
    with pytest.raises(ValueError, match="rank"):
        pka.paged_attn_forward(plan, q[0], k, v, 0.125)
    with pytest.raises(TypeError):
        pka.paged_attn_forward(plan, q, [[0.0]], v, 0.125)             # not a tensor
    with pytest.raises(ValueError, match="uploaded"):                  # everything else fine
        pka.paged_attn_forward(plan, q, k, v, 0.125)
    with pytest.raises(ValueError, match="uploaded"):
        pka.paged_attn_plan_advance(plan)
    with pytest.raises(ValueError, match="uploaded"):
        pka.paged_kv_store(plan, q, q, k, v)
    with pytest.raises(ValueError, match="rank"):
        pka.paged_kv_store(plan, q[0], q, k, v)


@pytest.mark.gpu
def test_refusals_with_an_uploaded_plan(cuda_device):
    dev = torch.device("cuda", 0)
    plan = _plan()
    plan.upload(dev)
    q, k, v = _tensors(dev)
    with pytest.raises(ValueError, match="is on"):                     # caches on the host
        pka.paged_attn_forward(plan, q, k.cpu(), v.cpu(), 0.125)
    with pytest.raises(ValueError, match="plan"):                      # pool size differs from the plan
        pka.paged_attn_forward(plan, q, k[:3].contiguous(), v[:3].contiguous(), 0.125)
    with pytest.raises(ValueError, match="queries"):                   # query count differs
        pka.paged_attn_forward(plan, q[:1].contiguous(), k, v, 0.125)
    with pytest.raises(ValueError, match="shape"):
        pka.paged_attn_forward(plan, q, k, v, 0.125, out=torch.empty(2, 4, 32, dtype=q.dtype, device=dev))
    buf = torch.zeros(2 * 4 * 64 * 2, dtype=q.dtype, device=dev)
    q_view, out_view = buf[:2 * 4 * 64].view(2, 4, 64), buf[2 * 4 * 64 - 64:-64].view(2, 4, 64)
    with pytest.raises(ValueError, match="overlaps"):                  # out shares storage with q
        pka.paged_attn_forward(plan, q_view, k, v, 0.125, out=out_view)
    ws = pka.make_workspace(plan, 4, 64, 2)
    with pytest.raises(ValueError, match="overlaps"):                  # out inside the workspace
        pka.paged_attn_forward_split(plan, q, k, v, 0.125, 2, workspace=ws,
                                     out=ws.view(torch.bfloat16)[:2 * 4 * 64].view(2, 4, 64))
    with pytest.raises(ValueError, match="one shared head"):           # MLA caches with two heads
        pka.paged_mla_forward(plan, q, q[:, :, :8].contiguous(), k, k[..., :8].contiguous(), 0.1)
    assert pka.device_status() == 0


def test_readme_calls_exist():
    """Every package function the README's usage snippet calls is exported."""
    import os
    import re
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    text = open(os.path.join(root, "README.md")).read()
    snippet = re.search(r"```python\n(.*?)```", text, flags=re.S).group(1)
    names = set(re.findall(r"\bpka\.(\w+)\(", snippet))
    assert {"paged_attn_plan", "paged_kv_store", "paged_attn_forward", "paged_mla_forward"} <= names
    for n in names:
        assert callable(getattr(pka, n, None)), f"README calls pka.{n}, which the package does not export"
    assert callable(getattr(pka.Plan, "stage", None))
