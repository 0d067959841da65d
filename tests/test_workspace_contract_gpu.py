"""The workspace and output contract of the C ABI, exercised with poisoned memory.

`include/fa.h` promises that the contents of a caller's workspace on entry do not matter and
that every output element is written. Each case here fills the workspace with 0xFF bytes (NaN
as fp32) and every output with NaN before the call, repeats the call several times, and checks
that all outputs are finite and agree with a run on zeroed memory:
- O and LSE bit for bit;
- dQ, dK and dV within the rounding of their fp32 reduction order.

The shapes cover the persistent d = 64 backward, the d = 128 backward with key padding, and
the decode kernel in both of its decompositions, including the join of heads cut between CTAs.
"""

import ctypes
import math

import pytest
import torch

import workloads
from io_aware_exact_04_gb300 import _lib

pytestmark = pytest.mark.gpu


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


TRAIN = [
    # B, H, N, d, causal, kv_len
    (4, 3, 1024, 64, True, None),
    (2, 4, 700, 128, False, [700, 333]),
    (3, 2, 520, 64, False, [1, 520, 0]),
]


@pytest.mark.parametrize("B,H,N,d,causal,kv_len", TRAIN)
def test_poisoned_workspace_and_outputs_training(gpu, B, H, N, d, causal, kv_len):
    lib = _lib.load("libfa.so")
    x = workloads.draw(B, H, N, d, seed=N + d)
    q, k, v, do = (x[n].to(gpu) for n in ("q", "k", "v", "do"))
    kv = None if kv_len is None else torch.tensor(kv_len, dtype=torch.int32, device=gpu)
    scale = 1.0 / math.sqrt(d)
    sp = ctypes.c_void_p(torch.cuda.current_stream(gpu).cuda_stream)
    wsb = int(lib.fa_backward_workspace_size(B, H, N, d))
    work = torch.empty(wsb, dtype=torch.uint8, device=gpu)

    def run(poison):
        fill = float("nan") if poison else 0.0
        o, dq, dk, dv = (torch.full_like(q, fill) for _ in range(4))
        lse = torch.full((B, H, N), fill, dtype=torch.float32, device=gpu)
        work.fill_(0xFF if poison else 0)
        assert lib.fa_forward_ex(_p(q), _p(k), _p(v), _p(o), _p(lse), B, H, N, d, scale, int(causal), _p(kv), sp) == 0
        assert lib.fa_backward_ex(_p(q), _p(k), _p(v), _p(o), _p(do), _p(lse), _p(dq), _p(dk), _p(dv), B, H, N, d,
                                  scale, int(causal), _p(kv), _p(work), wsb, sp) == 0
        torch.cuda.synchronize(gpu)
        detail = (ctypes.c_int * 4)()
        assert lib.fa_get_last_device_status_detail(sp, detail) == 0, list(detail)
        return {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}

    clean = run(False)
    for _ in range(4):
        got = run(True)
        for n, t in got.items():
            # LSE is -inf for rows without a valid key; everything else is finite
            assert not torch.isnan(t).any(), n
            assert torch.isfinite(t).all() or n == "lse", n
        assert torch.equal(got["o"], clean["o"])
        assert torch.equal(got["lse"], clean["lse"])
        for n in ("dq", "dk", "dv"):
            diff = float((got[n].float() - clean[n].float()).abs().max())
            assert diff <= 1e-2 * float(clean[n].float().abs().max()) + 1e-6, (n, diff)


DECODE = [
    # B, H, N_q, N_k, d, kv_len, n_split
    (8, 12, 1, 8192, 64, None, 1),       # whole heads a CTA
    (4, 3, 2, 5000, 64, None, 8),        # heads cut between CTAs: join kernel
    (5, 4, 4, 3000, 128, [3000, 1, 0, 2500, 129], 3),  # key padding, an empty batch: join kernel
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,kv_len,n_split", DECODE)
def test_poisoned_workspace_and_outputs_decode(gpu, B, H, Nq, Nk, d, kv_len, n_split):
    lib = _lib.load("libfa.so")
    x = workloads.draw(B, H, Nq, d, seed=Nk + n_split, Nk=Nk)
    q, k, v = (x[n].to(gpu) for n in ("q", "k", "v"))
    kv = None if kv_len is None else torch.tensor(kv_len, dtype=torch.int32, device=gpu)
    scale = 1.0 / math.sqrt(d)
    sp = ctypes.c_void_p(torch.cuda.current_stream(gpu).cuda_stream)
    wsb = int(lib.fa_forward_split_workspace_size(B, H, Nq, d, n_split))
    work = torch.empty(wsb, dtype=torch.uint8, device=gpu)

    def run(poison):
        fill = float("nan") if poison else 0.0
        o = torch.full_like(q, fill)
        lse = torch.full((B, H, Nq), fill, dtype=torch.float32, device=gpu)
        work.fill_(0xFF if poison else 0)
        assert lib.fa_forward_split(_p(q), _p(k), _p(v), _p(o), _p(lse), B, H, Nq, Nk, d, scale, 1, _p(kv), n_split,
                                    _p(work), wsb, sp) == 0
        torch.cuda.synchronize(gpu)
        return o, lse

    o0, l0 = run(False)
    for _ in range(4):
        o1, l1 = run(True)
        assert not torch.isnan(o1).any() and not torch.isnan(l1).any()
        assert torch.equal(o1, o0)
        assert torch.equal(l1, l0)
