"""Analytic training-memory model: stored attention matrices vs running statistics.

Restates the memory accounting of "FlashAttention Algorithm > Recomputation
Strategy" (section "Why Recomputation Makes Sense", code cell In[17] and its
printed table Out[18]) as used by the benchmark to print, next to the measured
peak activation memory, what a materialising implementation would store.

Per layer, with n tokens, model width d_model, h heads and b bytes/element:
  standard  = 2 * n^2 * h * b          (scores and softmax weights, every head)
            + 4 * n * d_model * b      (Q, K, V, O)
  recompute = 4 * n * d_model * b      (Q, K, V, O)
            + 2 * n * h * b            (two per-row statistics, m and l, per head)
Totals multiply by the layer count; GB means 1e9 bytes.
"""

from __future__ import annotations

from typing import Dict


def attention_matrix_bytes(n: int, dtype_bytes: int = 2) -> int:
    """Bytes of one n x n attention matrix (one head, one layer)."""
    return n * n * dtype_bytes


def training_memory(n: int, d_model: int, heads: int, layers: int, dtype_bytes: int = 2) -> Dict[str, float]:
    """Memory of stored attention state for the whole stack, both schemes."""
    matrices = 2 * n * n * heads * dtype_bytes
    qkvo = 4 * n * d_model * dtype_bytes
    stats = 2 * n * heads * dtype_bytes
    standard = layers * (matrices + qkvo)
    recompute = layers * (qkvo + stats)
    return {
        "standard_bytes": standard,
        "recompute_bytes": recompute,
        "standard_gb": standard / 1e9,
        "recompute_gb": recompute / 1e9,
        "savings_pct": 100.0 * (standard - recompute) / standard,
        "matrices_gb": layers * matrices / 1e9,
    }


def format_row(n: int, r: Dict[str, float]) -> str:
    """One line in the layout of the printed table (Out[18])."""
    return (f"{n:>10,} {r['standard_gb']:>11.2f}G {r['recompute_gb']:>11.3f}G "
            f"{r['savings_pct']:>9.1f}% {r['matrices_gb']:>13.2f}G")


def recompute_activation_bytes_per_row(d: int) -> int:
    """Bytes per (head, query row) that this library's fwd+bwd keeps besides
    the inputs and the gradients: O (bf16), LSE (fp32), D (fp32) and the fp32
    dQ accumulator."""
    return 2 * d + 4 + 4 + 4 * d
