"""The example GPT-2-small stack (examples/gpt2_layers.py): its attention through the
library against the same stack with plain PyTorch attention, and the checkpointed
(recomputing) run against the stored one."""

import pytest
import torch

pytestmark = pytest.mark.gpu


def _rel(a, b):
    return float((a.float() - b.float()).abs().max()) / max(float(b.float().abs().max()), 1e-6)


def _grads(model):
    return {n: p.grad.detach().clone() for n, p in model.named_parameters()}


def test_library_attention_matches_plain_attention_in_the_stack(gpu):
    from examples import gpt2_layers as m
    model, x = m.make(layers=2, batch=2, seq=256, device=gpu, seed=1)
    loss_lib = m.step(model, x, recompute=False, attn=m.library_attention)
    g_lib = _grads(model)
    loss_ref = m.step(model, x, recompute=False, attn=m.plain_attention)
    g_ref = _grads(model)
    assert abs(float(loss_lib) - float(loss_ref)) <= 2e-2 * abs(float(loss_ref))
    for n in g_ref:
        assert _rel(g_lib[n], g_ref[n]) < 5e-2, n


def test_checkpointed_stack_matches_stored(gpu):
    from examples import gpt2_layers as m
    model, x = m.make(layers=3, batch=2, seq=384, device=gpu, seed=2)
    loss_a = m.step(model, x, recompute=False)
    g_a = _grads(model)
    loss_b = m.step(model, x, recompute=True)
    g_b = _grads(model)
    assert float(loss_a) == float(loss_b)  # the forward is bitwise repeatable
    for n in g_a:
        assert _rel(g_b[n], g_a[n]) < 2e-2, n
