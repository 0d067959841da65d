"""Scores that grow along the keys, so that the running maxima actually move.

The forward keeps a row's reference maximum until a later key tile's scores exceed it by more
than 2^8 (in the base-2 domain); then it rescales O and the normaliser and moves the
reference. The training kernels do that per query row in TMEM and the decode kernel per lane.
Seeded normal inputs almost never trigger it after a row's first key tile. Here the keys'
norms ramp up along the sequence (key j scaled by 1 + a j / N_k: a = 3, or 12 over the long
key ranges of the inference cases) and the queries are scaled by 3, so later key tiles keep
overtaking the reference. A host-side count first checks, in the exact scores, that the inputs
do force many moves of the reference; then every path that keeps a running maximum is
compared with the fp64 oracle.
"""

import math

import numpy as np
import pytest
import torch

import workloads
from io_aware_exact_04_gb300 import api
from oracle import ref
from tests.parity_util import assert_within, compare, f64, run_gpu

pytestmark = pytest.mark.gpu

LOG2E = 1.4426950408889634


def _growing(B, H, N, d, seed, Nk=None, slope=3.0):
    x = workloads.draw(B, H, N, d, seed=seed, Nk=Nk)
    nk = x["k_f32"].shape[2]
    ramp = 1.0 + slope * torch.arange(nk, dtype=torch.float32) / nk
    q = x["q_f32"] * 3.0
    k = x["k_f32"] * ramp[None, None, :, None]
    x["q"], x["k"] = q.to(torch.bfloat16), k.to(torch.bfloat16)
    return x


def _moves(x, scale, causal):
    """(moves, tiles): over every head and query row, the key tiles (of 128) after the row's
    first one, and how many of them have a row maximum more than 2^8 above the reference."""
    q, k = f64(x["q"]), f64(x["k"])
    moves = later = 0
    for b in range(q.shape[0]):
        for h in range(q.shape[1]):
            s = (q[b, h] @ k[b, h].T) * scale * LOG2E
            nq, nk = s.shape
            if causal:
                s = np.where(np.arange(nk)[None, :] <= np.arange(nq)[:, None] + nk - nq, s, -np.inf)
            tmax = np.stack([s[:, j0:j0 + 128].max(axis=1) for j0 in range(0, nk, 128)], axis=1)
            for row in tmax:
                ref_m = -np.inf
                for m in row:
                    if m == -np.inf:
                        continue
                    if ref_m == -np.inf:
                        ref_m = m
                        continue
                    later += 1
                    if m > ref_m + 8.0:
                        moves += 1
                        ref_m = m
    return moves, later


TRAIN = [
    # B, H, N, d, causal
    (1, 2, 1000, 64, True),    # the persistent d = 64 forward
    (2, 2, 600, 64, False),
    (1, 2, 1500, 64, True),    # the per-item d = 64 forward (rows past 1024)
    (1, 2, 700, 128, True),    # d = 128: P written over S
]


@pytest.mark.parametrize("B,H,N,d,causal", TRAIN)
def test_moving_maxima_forward_and_backward_match_oracle(gpu, B, H, N, d, causal):
    x = _growing(B, H, N, d, seed=N + d)
    scale = 1 / math.sqrt(d)
    moves, later = _moves(x, scale, causal)
    assert moves >= 10 and moves >= 0.05 * later, (moves, later)  # the path under test does run
    g = run_gpu(x, causal, gpu)
    r = ref.attention(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["do"]), scale=scale, causal=causal)
    assert_within({n: compare(n, f64(g[n]), r[n]) for n in ("o", "lse", "dq", "dk", "dv")})


DECODE = [
    # B, H, N_q, N_k, d, n_split
    (2, 3, 1, 5000, 64, 1),    # whole heads a CTA
    (2, 3, 2, 5000, 64, 8),    # heads cut between CTAs, joined
    (2, 2, 4, 3000, 128, 3),   # d = 128
    (1, 2, 300, 3000, 64, 3),  # the split forward of query tiles and its join
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,n_split", DECODE)
def test_moving_maxima_inference_forward_matches_oracle(gpu, B, H, Nq, Nk, d, n_split):
    x = _growing(B, H, Nq, d, seed=Nk + d, Nk=Nk, slope=12.0)
    scale = 1 / math.sqrt(d)
    moves, later = _moves(x, scale, True)
    assert moves >= 10 and moves >= 0.05 * later, (moves, later)
    q, k, v = (x[n].to(gpu) for n in ("q", "k", "v"))
    o, lse = api.forward_split(q, k, v, causal=True, n_split=n_split, with_lse=True)
    torch.cuda.synchronize(gpu)
    code, detail = api.device_status(gpu)
    assert code == 0, detail
    r = ref.attention(f64(x["q"]), f64(x["k"]), f64(x["v"]), scale=scale, causal=True, backward=False)
    assert_within({"o": compare("o", f64(o), r["o"]), "lse": compare("lse", f64(lse), r["lse"])})


@pytest.mark.parametrize("d", [64, 128])
def test_moving_maxima_packed_sequences_match_oracle(gpu, d):
    H, lens = 2, [500, 700, 90]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    full = workloads.draw(1, H, int(cu[-1]), d, seed=11 + d)
    # keys ramp up within each sequence
    ramp = torch.cat([1.0 + 3.0 * torch.arange(n, dtype=torch.float32) / n for n in lens])
    q = (full["q_f32"][0] * 3.0).to(torch.bfloat16)
    k = (full["k_f32"][0] * ramp[None, :, None]).to(torch.bfloat16)
    v, do = full["v"][0], full["do"][0]
    cu_d = torch.tensor(cu, device=gpu)
    qg, kg, vg, dog = (t.to(gpu) for t in (q, k, v, do))
    o, lse = api.forward_varlen(qg, kg, vg, cu_d, max(lens), causal=True)
    dq, dk, dv = api.backward_varlen(qg, kg, vg, o, dog, lse, cu_d, max(lens), causal=True)
    torch.cuda.synchronize(gpu)
    code, detail = api.device_status(gpu)
    assert code == 0, detail
    r = ref.attention_varlen(f64(q), f64(k), f64(v), f64(do), cu, scale=1 / math.sqrt(d), causal=True)
    assert_within({n: compare(n, f64(t), r[n]) for n, t in
                   (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))})
