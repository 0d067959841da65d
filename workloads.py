"""Seeded synthetic attention workloads (shapes, value distributions, draw order).

This module holds no attention arithmetic: it only names the workloads and
draws their random inputs, so that the fp64 oracle and the CUDA path can be
fed the very same bf16 tensors.

Workload shapes follow the end-to-end settings that the FlashAttention
practice record cites (GPT-2, BERT-large; "Why recomputation is cheaper here
than storing") and the GPT-2 memory-table configuration (d_model 768, 12
heads) of "FlashAttention Algorithm > Recomputation Strategy", In[17]/Out[18].
No dataset or trained weight is involved: every tensor is i.i.d. Gaussian.

Draw recipe (one CPU ``torch.Generator`` seeded with ``seed``):
  1. q, k, v, dO drawn in that order as fp32 standard normals, q and dO
     ``[B, H, N, d]``, k and v ``[B, H, N_k, d]`` (N_k = N for every named
     workload; the tests of unequal lengths set it);
  2. q and k multiplied by ``qk_scale`` (0.5 for the head-dim-128 workload);
  3. for key-padded workloads, per-sequence valid key counts drawn from the
     same generator as integers uniform in ``[len_lo, len_hi]`` inclusive;
  4. q, k, v, dO rounded to bf16 (round to nearest even).
"""

from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    qk_scale: float = 1.0
    len_lo: Optional[int] = None  # key padding: valid lengths uniform in [len_lo, len_hi]
    len_hi: Optional[int] = None
    Nk: Optional[int] = None      # key rows when they differ from the N query rows
    infer: bool = False           # forward only, split keys (inference): no backward, no LSE
    packed: bool = False          # the padded draw's valid rows packed per head: [H, T, d], cu_seqlens

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def padded(self) -> bool:
        return self.len_lo is not None

    @property
    def nk(self) -> int:
        return self.N if self.Nk is None else self.Nk

    def describe(self) -> str:
        s = f"{self.name}: B={self.B} H={self.H} N={self.N} d={self.d} " + (
            "causal" if self.causal else "non-causal")
        if self.Nk is not None:
            s += f", N_k={self.Nk} (causal queries aligned with the last keys)"
        if self.infer:
            s += ", forward only (inference, split keys)"
        if self.packed:
            s += ", sequences packed to their lengths ([H, T, d], cu_seqlens)"
        if self.padded:
            s += f", key padding len~U[{self.len_lo},{self.len_hi}]"
        if self.qk_scale != 1.0:
            s += f", q,k x{self.qk_scale}"
        return s


WORKLOADS: Dict[str, Workload] = {
    w.name: w
    for w in [
        Workload("tiny", 1, 1, 128, 64, False),
        Workload("gpt2", 8, 12, 1024, 64, True),
        Workload("bert", 16, 16, 512, 64, False, len_lo=128, len_hi=512),
        Workload("d128", 2, 16, 4096, 128, True, qk_scale=0.5),
        Workload("long2048", 1, 12, 2048, 64, True),
        Workload("long8192", 1, 12, 8192, 64, True),
        Workload("long16384", 1, 12, 16384, 64, True),
        Workload("long32768", 1, 12, 32768, 64, True),
        # unequal lengths: 1024 new queries over 4096 keys (3072 earlier positions + themselves)
        Workload("prefill1024_kv4096", 8, 12, 1024, 64, True, Nk=4096),
        # inference: one new query per sequence over 8192 keys (forward only, split keys)
        Workload("decode_kv8192", 8, 12, 1, 64, True, Nk=8192, infer=True),
        # the bert draw with each sequence's valid rows packed (no padding rows computed)
        Workload("bert_packed", 16, 16, 512, 64, False, len_lo=128, len_hi=512, packed=True),
    ]
}


def draw(B: int, H: int, N: int, d: int, *, seed: int = 0, qk_scale: float = 1.0,
         len_range: Optional[tuple] = None, Nk: Optional[int] = None) -> Dict[str, Optional[torch.Tensor]]:
    """Draw q, k, v, dO (bf16, CPU) and optional kv_len (int32 ``[B]``): q and dO are
    ``[B,H,N,d]``, k and v ``[B,H,Nk,d]`` (Nk defaults to N)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    shape = (B, H, N, d)
    kshape = (B, H, N if Nk is None else Nk, d)
    q = torch.randn(shape, generator=g, dtype=torch.float32)
    k = torch.randn(kshape, generator=g, dtype=torch.float32)
    v = torch.randn(kshape, generator=g, dtype=torch.float32)
    do = torch.randn(shape, generator=g, dtype=torch.float32)
    if qk_scale != 1.0:
        q = q * qk_scale
        k = k * qk_scale
    kv_len = None
    if len_range is not None:
        lo, hi = len_range
        kv_len = torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int64).to(torch.int32)
    return {
        "q": q.to(torch.bfloat16),
        "k": k.to(torch.bfloat16),
        "v": v.to(torch.bfloat16),
        "do": do.to(torch.bfloat16),
        "kv_len": kv_len,
        "q_f32": q, "k_f32": k, "v_f32": v, "do_f32": do,
    }


def make_inputs(w: Workload, seed: int = 0) -> Dict[str, Optional[torch.Tensor]]:
    rng = (w.len_lo, w.len_hi) if w.padded else None
    return draw(w.B, w.H, w.N, w.d, seed=seed, qk_scale=w.qk_scale, len_range=rng, Nk=w.Nk)


def pack(x: Dict[str, Optional[torch.Tensor]]) -> Dict[str, torch.Tensor]:
    """The valid rows of a key-padded draw, packed per head: q, k, v, dO [H, T, d] (sequence b's
    first kv_len[b] rows, back to back) and cu_seqlens int32 [B + 1]."""
    kv = x["kv_len"].to(torch.int64)
    cu = torch.zeros(kv.numel() + 1, dtype=torch.int64)
    cu[1:] = torch.cumsum(kv, 0)
    out = {"cu_seqlens": cu.to(torch.int32)}
    for n in ("q", "k", "v", "do"):
        t = x[n]  # [B, H, N, d]
        out[n] = torch.cat([t[b, :, :int(kv[b])] for b in range(t.shape[0])], dim=1).contiguous()
    return out


def visible_pairs(nq: int, nk: int, causal: bool, kv: Optional[int] = None) -> float:
    """Query-key pairs of one head as FLOP counts take them: N_q * kv without a causal
    mask; with one (query i keeps keys j <= i + N_k - N_q and j < kv) the area under that
    bound over the rows, so that the diagonal counts half, as in the usual c = 1/2."""
    kv = nk if kv is None else kv
    if not causal:
        return float(nq * kv)
    off = nk - nq
    x0 = max(0.0, float(-off))                   # first row that keeps a key
    x1 = min(max(float(kv - off), x0), float(nq))  # rows past x1 keep all kv keys
    return ((x1 + off) ** 2 - (x0 + off) ** 2) / 2 + kv * (nq - x1)


def flop_counts(w: Workload, kv_len: Optional[torch.Tensor] = None) -> Dict[str, float]:
    """Matmul FLOPs of one fwd+bwd over the workload.

    Per head: fwd 4*P*d (QK^T and PV), bwd nominal 8*P*d (dV, dP, dK, dQ) and
    recompute 2*P*d (QK^T again), with P = visible_pairs (c * N * N_k for square
    causal masks, c = 1/2 with the diagonal counted half, the usual convention;
    N_k the valid key count).
    """
    if kv_len is not None:
        pairs = sum(visible_pairs(w.N, w.nk, w.causal, int(x)) for x in kv_len.tolist()) * w.H
    else:
        pairs = visible_pairs(w.N, w.nk, w.causal) * w.B * w.H
    base = pairs * w.d
    return {"fwd": 4 * base, "bwd_nominal": 8 * base, "bwd_recompute": 2 * base,
            "fwd_bwd_nominal": 12 * base, "fwd_bwd_executed": 14 * base}
