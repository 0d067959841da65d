"""fp64 CPU oracle for exact softmax attention, forward and backward.

TEST INFRASTRUCTURE. Only the test suite, the smoke check and the benchmark's
CPU-baseline leg may import this module. The CUDA path never calls it, and it
calls nothing from the CUDA path.

What it computes is the plain definition, written out: it materialises the full
score matrix S and the probability matrix P of each head, in float64, exactly
the N x N matrices that the tiled method avoids storing.

  Forward (practice record "Why recomputation is cheaper here than storing",
  first paragraph: scores S, softmax, then the product with V; the saved
  per-row statistics are the running maximum m and normaliser l, handbook
  "FlashAttention Algorithm > Recomputation Strategy", section "What Gets
  Stored vs Recomputed"):
      S   = s * Q K^T             masked entries set to -inf
      m   = rowmax S
      l   = rowsum exp(S - m)
      P   = exp(S - m) / l
      LSE = m + ln l              (m and l folded into one natural-log value)
      O   = P V

  Backward (the gradient of the scalar L = sum(O * dO) through the forward
  above, i.e. the textbook softmax Jacobian; the pages name only that the
  gradients are formed block by block from recomputed S and P):
      D  = rowsum(dO * O)
      dV = P^T dO
      dP = dO V^T
      dS = P * (dP - D)
      dQ = s * dS K
      dK = s * dS^T Q

Masks: causal keeps key j for query i iff j <= i + (N_k - N_q): the N_q query
rows stand for the last N_q positions of the N_k keys' sequence, so that for
N_q = N_k this is j <= i (diagonal kept); key padding keeps key j iff
j < kv_len. A row whose keys are all masked (kv_len = 0, or a causal row before
the first key when N_q > N_k) has O = 0, LSE = -inf and contributes nothing to
any gradient.

Every function takes float64 numpy arrays (callers pass the bf16-rounded
inputs upcast to float64). Library primitives used as single steps: numpy
matmul, exp, log, max, sum.
"""

from __future__ import annotations

from typing import Dict, Iterable, Optional

import numpy as np


def keep_mask(rows: np.ndarray, cols: np.ndarray, causal: bool, kv_len: Optional[int],
              offset: int = 0) -> np.ndarray:
    """Boolean [len(rows), len(cols)]: True where query row i may attend to key j.

    ``offset`` = N_k - N_q aligns the query rows with the last keys (causal only)."""
    i = np.asarray(rows)[:, None]
    j = np.asarray(cols)[None, :]
    keep = np.ones((i.shape[0], j.shape[1]), dtype=bool)
    if causal:
        keep &= j <= i + int(offset)
    if kv_len is not None:
        keep &= j < int(kv_len)
    return keep


def scores(q: np.ndarray, k: np.ndarray, scale: float, causal: bool,
           kv_len: Optional[int], rows: np.ndarray) -> np.ndarray:
    """S = s * Q[rows] K^T with masked entries at -inf."""
    s_mat = scale * (q[rows] @ k.T)
    s_mat[~keep_mask(rows, np.arange(k.shape[0]), causal, kv_len, k.shape[0] - q.shape[0])] = -np.inf
    return s_mat


def softmax_stats(s_mat: np.ndarray):
    """Row softmax of a masked score matrix: returns (P, LSE, m, l)."""
    m = s_mat.max(axis=1)
    empty = ~np.isfinite(m)
    m_safe = np.where(empty, 0.0, m)
    e = np.exp(s_mat - m_safe[:, None])  # exp(-inf) = 0 on masked entries
    l_row = e.sum(axis=1)
    l_safe = np.where(empty, 1.0, l_row)
    p = e / l_safe[:, None]
    with np.errstate(divide="ignore"):
        lse = np.where(empty, -np.inf, m_safe + np.log(l_safe))
    return p, lse, m, l_row


def probs(q, k, scale, causal, kv_len=None, rows=None) -> np.ndarray:
    """The attention matrix P of one head (rows subset optional)."""
    rows = np.arange(q.shape[0]) if rows is None else np.asarray(rows)
    return softmax_stats(scores(q, k, scale, causal, kv_len, rows))[0]


def head_forward(q, k, v, scale: float, causal: bool, kv_len: Optional[int] = None,
                 rows: Optional[Iterable[int]] = None):
    """One head: returns (O[rows], LSE[rows]). Each row is independent of the others."""
    rows = np.arange(q.shape[0]) if rows is None else np.asarray(list(rows), dtype=np.int64)
    p, lse, _, _ = softmax_stats(scores(q, k, scale, causal, kv_len, rows))
    return p @ v, lse


def head_backward(q, k, v, do, scale: float, causal: bool, kv_len: Optional[int] = None,
                  row_block: Optional[int] = None) -> Dict[str, np.ndarray]:
    """One head, forward and backward from the definition.

    Returns o, lse, D, dq, dk, dv. ``row_block`` splits the query rows into
    consecutive groups so that S and P are materialised one group at a time
    (memory, not arithmetic: every row's S, P, O, D, dS and dQ depend on that
    row alone, and dK, dV are sums over rows, here accumulated group by group).
    """
    n = q.shape[0]
    row_block = n if row_block is None else max(1, int(row_block))
    o = np.zeros_like(q)
    lse = np.zeros(n)
    dd = np.zeros(n)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for r0 in range(0, n, row_block):
        rows = np.arange(r0, min(n, r0 + row_block))
        p, lse_r, _, _ = softmax_stats(scores(q, k, scale, causal, kv_len, rows))
        o_r = p @ v
        do_r = do[rows]
        d_r = (do_r * o_r).sum(axis=1)          # D = rowsum(dO * O)
        dv += p.T @ do_r                        # dV = P^T dO
        dp = do_r @ v.T                         # dP = dO V^T
        ds = p * (dp - d_r[:, None])            # dS = P * (dP - D)
        dq[rows] = scale * (ds @ k)             # dQ = s dS K
        dk += scale * (ds.T @ q[rows])          # dK = s dS^T Q
        o[rows] = o_r
        lse[rows] = lse_r
        dd[rows] = d_r
    return {"o": o, "lse": lse, "D": dd, "dq": dq, "dk": dk, "dv": dv}


def head_sampled(q, k, v, do, scale: float, causal: bool, kv_len: Optional[int],
                 rows: Iterable[int], keys: Iterable[int], row_block: int = 2048) -> Dict[str, np.ndarray]:
    """Selected outputs of one head, each from the definition, for sequences too
    long to hold one head's S in memory.

    O, LSE, D and dQ of query row i depend on row i of S only. dK and dV of key
    j are sums over all query rows of column j of P and dS, which need every
    row's LSE and D; those come from a forward pass over consecutive groups of
    ``row_block`` rows (memory only: each row is computed on its own).
    """
    n = q.shape[0]
    rows = np.asarray(list(rows), dtype=np.int64)
    keys = np.asarray(list(keys), dtype=np.int64)
    lse = np.zeros(n)
    dd = np.zeros(n)
    for r0 in range(0, n, row_block):
        rr = np.arange(r0, min(n, r0 + row_block))
        p, lse_r, _, _ = softmax_stats(scores(q, k, scale, causal, kv_len, rr))
        lse[rr] = lse_r
        dd[rr] = (do[rr] * (p @ v)).sum(axis=1)     # D = rowsum(dO * O)
    # rows: O, LSE, dQ from row i of S, P, dP, dS
    p, _, _, _ = softmax_stats(scores(q, k, scale, causal, kv_len, rows))
    o_rows = p @ v
    dp = do[rows] @ v.T
    ds = p * (dp - dd[rows][:, None])
    dq_rows = scale * (ds @ k)
    # keys: column j of S, P, dP, dS over all rows
    s_cols = scale * (q @ k[keys].T)                                  # [n, len(keys)]
    keep = keep_mask(np.arange(n), keys, causal, kv_len, k.shape[0] - n)
    with np.errstate(invalid="ignore"):
        p_cols = np.where(keep & np.isfinite(lse)[:, None], np.exp(s_cols - lse[:, None]), 0.0)
    dp_cols = do @ v[keys].T
    ds_cols = p_cols * (dp_cols - dd[:, None])
    dv_keys = p_cols.T @ do
    dk_keys = scale * (ds_cols.T @ q)
    return {"o": o_rows, "lse": lse[rows], "D": dd[rows], "dq": dq_rows,
            "dk": dk_keys, "dv": dv_keys, "lse_all": lse, "D_all": dd}


def head_intermediates(q, k, v, do, scale, causal, kv_len=None) -> Dict[str, np.ndarray]:
    """S, P, dP, dS of one head (whole matrices), for invariant checks on small inputs."""
    rows = np.arange(q.shape[0])
    s_mat = scores(q, k, scale, causal, kv_len, rows)
    p, lse, m, l_row = softmax_stats(s_mat)
    o = p @ v
    d_r = (do * o).sum(axis=1)
    dp = do @ v.T
    ds = p * (dp - d_r[:, None])
    return {"S": s_mat, "P": p, "m": m, "l": l_row, "lse": lse, "o": o, "D": d_r, "dP": dp, "dS": ds}


def attention(q, k, v, do=None, *, scale: float, causal: bool, kv_len=None,
              heads: Optional[Iterable] = None, row_block: Optional[int] = None,
              backward: bool = True) -> Dict[str, np.ndarray]:
    """Batched driver over float64 arrays: q, do [B, H, N_q, d]; k, v [B, H, N_k, d].

    ``kv_len`` is None or a length-B integer array. ``heads`` optionally lists
    (b, h) pairs; outputs are then stacked in that order as [len(heads), N, ...].
    Without ``heads`` outputs have the input's [B, H, ...] layout.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, H, N, d = q.shape
    pairs = [(b, h) for b in range(B) for h in range(H)] if heads is None else list(heads)
    out = {key: [] for key in (["o", "lse", "D", "dq", "dk", "dv"] if backward else ["o", "lse"])}
    for b, h in pairs:
        kl = None if kv_len is None else int(kv_len[b])
        if backward:
            r = head_backward(q[b, h], k[b, h], v[b, h], np.asarray(do[b, h], dtype=np.float64),
                              scale, causal, kl, row_block)
        else:
            o, lse = head_forward(q[b, h], k[b, h], v[b, h], scale, causal, kl)
            r = {"o": o, "lse": lse}
        for key in out:
            out[key].append(r[key])
    res = {key: np.stack(val) for key, val in out.items()}
    if heads is None:
        res = {key: val.reshape((B, H) + val.shape[1:]) for key, val in res.items()}
    return res


def attention_varlen(q, k, v, do, cu_seqlens, *, scale: float, causal: bool,
                     backward: bool = True) -> Dict[str, np.ndarray]:
    """Packed sequences: q, k, v, do are [H, T, d] float64 arrays and sequence b holds rows
    cu_seqlens[b] .. cu_seqlens[b + 1] of every head. Each sequence is its own attention
    problem (no query of one sequence sees a key of another); outputs keep the packed
    layout: o, dq, dk, dv [H, T, d]; lse, D [H, T]."""
    q = np.asarray(q, dtype=np.float64)
    H, T, d = q.shape
    cu = [int(x) for x in cu_seqlens]
    keys = ["o", "lse", "D", "dq", "dk", "dv"] if backward else ["o", "lse"]
    out = {key: np.zeros((H, T, d) if key in ("o", "dq", "dk", "dv") else (H, T)) for key in keys}
    for h in range(H):
        for s0, s1 in zip(cu[:-1], cu[1:]):
            if s1 <= s0:
                continue
            sl = slice(s0, s1)
            if backward:
                r = head_backward(q[h, sl], k[h, sl], v[h, sl], np.asarray(do[h, sl], dtype=np.float64), scale, causal)
            else:
                o, lse = head_forward(q[h, sl], k[h, sl], v[h, sl], scale, causal)
                r = {"o": o, "lse": lse}
            for key in keys:
                out[key][h, sl] = r[key]
    return out
