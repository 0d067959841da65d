"""A synthetic GPT-2-small stack run forward and backward with random weights.

Twelve blocks of d_model 768, 12 heads of 64, an MLP of 3072 and causal attention. Attention
goes through the library's exact tiled kernels, which keep only O and one LSE per row for
the backward pass. The stack runs either storing every block's activations or with each
block checkpointed: its forward pass runs again during the backward pass, and only block
inputs are kept. The latter is the recompute-based setting of the practice record's
end-to-end results ("Why recomputation is cheaper here than storing"). No dataset or
trained weight is involved: inputs and weights are seeded Gaussians.

    python examples/gpt2_layers.py [--layers 12] [--batch 8] [--seq 1024] [--steps 10]

One JSON line per mode (stored, checkpointed): ms per fwd+bwd step, tokens per second,
and peak memory above what stays resident between steps (weights, input, gradients).
"""

from __future__ import annotations

import argparse
import json
import math
import os
import sys

import torch
import torch.nn.functional as F
from torch.utils.checkpoint import checkpoint

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

from io_aware_exact_04_gb300 import api  # noqa: E402


def library_attention(q, k, v):
    """[B, H, N, d] bf16 -> O: the library's exact attention (causal)."""
    return api.attention(q, k, v, causal=True)


def plain_attention(q, k, v):
    """The same attention in plain PyTorch, fp32 scores (for comparison in tests only)."""
    n = q.shape[2]
    s = (q.float() @ k.float().transpose(-1, -2)) / math.sqrt(q.shape[-1])
    s = s.masked_fill(torch.ones(n, n, dtype=torch.bool, device=q.device).triu(1), float("-inf"))
    return (torch.softmax(s, dim=-1) @ v.float()).to(q.dtype)


class Block(torch.nn.Module):
    def __init__(self, d_model=768, heads=12, mlp=3072):
        super().__init__()
        self.heads = heads
        self.ln1 = torch.nn.LayerNorm(d_model)
        self.qkv = torch.nn.Linear(d_model, 3 * d_model)
        self.proj = torch.nn.Linear(d_model, d_model)
        self.ln2 = torch.nn.LayerNorm(d_model)
        self.fc = torch.nn.Linear(d_model, mlp)
        self.fc2 = torch.nn.Linear(mlp, d_model)

    def forward(self, x, attn):
        B, N, C = x.shape
        h = self.heads
        qkv = self.qkv(self.ln1(x)).view(B, N, 3, h, C // h).permute(2, 0, 3, 1, 4)  # [3, B, H, N, d]
        q, k, v = (t.contiguous() for t in qkv)
        o = attn(q, k, v).transpose(1, 2).reshape(B, N, C)
        x = x + self.proj(o)
        return x + self.fc2(F.gelu(self.fc(self.ln2(x))))


class Stack(torch.nn.Module):
    def __init__(self, layers=12, **kw):
        super().__init__()
        self.blocks = torch.nn.ModuleList(Block(**kw) for _ in range(layers))

    def forward(self, x, attn=library_attention, recompute=False):
        for blk in self.blocks:
            x = checkpoint(blk, x, attn, use_reentrant=False) if recompute else blk(x, attn)
        return x


def make(layers, batch, seq, device, seed=0):
    g = torch.Generator(device="cpu").manual_seed(seed)
    model = Stack(layers)
    with torch.no_grad():  # Linear weights N(0, 0.02^2), LayerNorm weights 1, biases 0
        for name, p in model.named_parameters():
            if p.dim() > 1:
                p.copy_(torch.randn(p.shape, generator=g) * 0.02)
            else:
                p.fill_(1.0 if name.split(".")[-2].startswith("ln") and name.endswith("weight") else 0.0)
    model = model.to(device=device, dtype=torch.bfloat16)
    x = torch.randn(batch, seq, 768, generator=g).to(device=device, dtype=torch.bfloat16)
    return model, x


def step(model, x, recompute, attn=library_attention):
    model.zero_grad(set_to_none=True)
    xi = x.detach().requires_grad_(True)
    out = model(xi, attn=attn, recompute=recompute)
    loss = out.float().pow(2).mean()
    loss.backward()
    return loss


def measure(layers, batch, seq, steps, recompute, device):
    model, x = make(layers, batch, seq, device)
    for _ in range(3):
        step(model, x, recompute)
    torch.cuda.synchronize(device)
    base = torch.cuda.memory_allocated(device)
    torch.cuda.reset_peak_memory_stats(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        step(model, x, recompute)
    e1.record()
    torch.cuda.synchronize(device)
    ms = e0.elapsed_time(e1) / steps
    peak = torch.cuda.max_memory_allocated(device) - base
    return {"mode": "checkpointed" if recompute else "stored", "layers": layers, "batch": batch, "seq": seq,
            "ms_per_step": ms, "tokens_per_s": batch * seq / (ms * 1e-3), "peak_bytes_above_resident": peak,
            "attention": "library (exact, tiled)", "dtype": "bf16", "data": "synthetic (seeded N(0,1))"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--layers", type=int, default=12)
    ap.add_argument("--batch", type=int, default=8)
    ap.add_argument("--seq", type=int, default=1024)
    ap.add_argument("--steps", type=int, default=10)
    args = ap.parse_args()
    dev = torch.device("cuda", 0)
    for recompute in (False, True):
        print(json.dumps(measure(args.layers, args.batch, args.seq, args.steps, recompute, dev)), flush=True)


if __name__ == "__main__":
    main()
