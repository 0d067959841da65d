"""The bounds-checked build (libfa_debug.so, include/fa_debug.h) on the GPU.

It stands in for a memory checker. The tests below show two things:
- On valid inputs none of its checks fires, and it computes what the oracle does. The shapes
  reach every kernel:
  - the persistent d = 64 forward and backward;
  - the per-item forward for long rows and for d = 128, and the d = 128 backward;
  - N_q != N_k;
  - packed sequences, forward and backward;
  - the split forward and its join;
  - the decode kernel in both decompositions, with its join.
- With the check slack (row extents taken down by one row), checks near the end of a tensor
  fail on memory that is really there (training at d = 64 and 128, packed sequences, decode). The call reports FA_ERR_DEVICE_CHECK with a site from
  fa_debug.h, and the CUDA context stays usable: the next call is clean and correct. Every
  access still stays inside the tensors, because a failed check only skips its access.
"""

import ctypes
import math

import numpy as np
import pytest
import torch

import workloads
from io_aware_exact_04_gb300 import _lib, api
from oracle import ref
from tests.parity_util import assert_within, check_all_heads, compare, f64

pytestmark = pytest.mark.gpu

SITES = range(100, 108)  # FA_DBG_META .. FA_DBG_TMEM


@pytest.fixture
def dbg(gpu, monkeypatch):
    """api's wrappers, routed to the debug build (its own status word included)."""
    lib = _lib.load("libfa_debug.so")
    monkeypatch.setattr(api, "_lib_fa", lambda: lib)
    assert lib.fa_debug_set_check_slack(0) == 0
    api.device_status(gpu)  # start from a clear word
    yield lib
    lib.fa_debug_set_check_slack(0)


TRAIN = [
    # B, H, Nq, Nk, d, causal, kv_len
    (2, 3, 300, 300, 64, True, [300, 77]),      # persistent d = 64 forward and backward
    (1, 2, 1300, 1300, 64, True, None),         # long rows: the per-item d = 64 forward
    (2, 2, 390, 390, 128, False, [390, 5]),     # d = 128 forward and backward, key padding
    (1, 2, 200, 1100, 64, True, None),          # N_q != N_k
    (2, 1, 130, 130, 128, True, [0, 130]),      # a batch with no valid key
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal,kv_len", TRAIN)
def test_no_check_fires_and_results_match_oracle(dbg, gpu, B, H, Nq, Nk, d, causal, kv_len):
    # check_all_heads runs api.forward / api.backward (now the debug build) and asserts that the
    # device status word is clear afterwards
    errs = check_all_heads(B, H, Nq, d, causal, kv_len, seed=Nq + d, device=gpu, Nk=Nk)
    assert_within(errs)


@pytest.mark.parametrize("d", [64, 128])
def test_packed_sequences_no_check_fires(dbg, gpu, d):
    H, lens = 2, [100, 257, 3, 130]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    full = workloads.draw(1, H, int(cu[-1]), d, seed=d)  # packed [H, T, d] tensors
    x = {n: full[n][0] for n in ("q", "k", "v", "do")}
    q, k, v, do = (x[n].to(gpu) for n in ("q", "k", "v", "do"))
    cu_d = torch.tensor(cu, device=gpu)
    o, lse = api.forward_varlen(q, k, v, cu_d, max(lens), causal=True)
    dq, dk, dv = api.backward_varlen(q, k, v, o, do, lse, cu_d, max(lens), causal=True)
    torch.cuda.synchronize(gpu)
    code, detail = api.device_status(gpu)
    assert code == 0, detail
    r = ref.attention_varlen(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["do"]), cu, scale=1 / math.sqrt(d),
                             causal=True)
    assert_within({n: compare(n, f64(t), r[n]) for n, t in
                   (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))})


SPLIT = [
    # B, H, Nq, Nk, d, kv_len, n_split
    (2, 2, 300, 2000, 64, [2000, 900], 3),   # split forward of query tiles, then its join
    (8, 12, 1, 3000, 64, None, 1),            # decode: whole heads a CTA
    (2, 3, 2, 5000, 64, None, 8),             # decode: heads cut between CTAs, then the join
    (3, 2, 4, 2100, 128, [2100, 1, 0], 3),    # decode d = 128, key padding, an empty batch
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,kv_len,n_split", SPLIT)
def test_split_and_decode_no_check_fires(dbg, gpu, B, H, Nq, Nk, d, kv_len, n_split):
    x = workloads.draw(B, H, Nq, d, seed=Nk + n_split, Nk=Nk)
    q, k, v = (x[n].to(gpu) for n in ("q", "k", "v"))
    kv = None if kv_len is None else torch.tensor(kv_len, dtype=torch.int32, device=gpu)
    o, lse = api.forward_split(q, k, v, causal=True, kv_len=kv, n_split=n_split, with_lse=True)
    torch.cuda.synchronize(gpu)
    code, detail = api.device_status(gpu)
    assert code == 0, detail
    r = ref.attention(f64(x["q"]), f64(x["k"]), f64(x["v"]), scale=1 / math.sqrt(d), causal=True,
                      kv_len=None if kv_len is None else np.asarray(kv_len), backward=False)
    assert_within({"o": compare("o", f64(o), r["o"]), "lse": compare("lse", f64(lse), r["lse"])})


def _reported_then_clean(gpu, run):
    """run() under a one-row check slack reports a device check; without it, all is clean."""
    lib = api._lib_fa()
    assert lib.fa_debug_set_check_slack(1) == 0
    run()
    torch.cuda.synchronize(gpu)
    code, detail = api.device_status(gpu)
    assert code == 6, detail                 # FA_ERR_DEVICE_CHECK
    assert detail[1] in SITES, detail
    assert api.device_status(gpu)[0] == 0    # reading the word cleared it
    assert lib.fa_debug_set_check_slack(0) == 0
    out = run()
    torch.cuda.synchronize(gpu)
    code, detail = api.device_status(gpu)
    assert code == 0, detail
    return out


@pytest.mark.parametrize("d", [64, 128])
def test_training_checks_fire_under_slack_and_context_survives(dbg, gpu, d):
    # 257 rows: the last 128-row tile starts on the last row, which the slack puts out of range
    B, H, N = 1, 2, 257
    x = workloads.draw(B, H, N, d, seed=7)
    q, k, v, do = (x[n].to(gpu) for n in ("q", "k", "v", "do"))

    def run():
        o, lse = api.forward(q, k, v, causal=True)
        return (o, lse) + tuple(api.backward(q, k, v, o, do, lse, causal=True))

    o, lse, dq, dk, dv = _reported_then_clean(gpu, run)
    r = ref.attention(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["do"]), scale=1 / math.sqrt(d), causal=True)
    assert_within({n: compare(n, f64(t), r[n]) for n, t in
                   (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))})


@pytest.mark.parametrize("d", [64, 128])
def test_packed_checks_fire_under_slack_and_context_survives(dbg, gpu, d):
    # packed sequences: the last sequence's rows end at the last row of each head's T rows
    H, lens = 2, [100, 257, 3, 130]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    full = workloads.draw(1, H, int(cu[-1]), d, seed=5 + d)
    x = {n: full[n][0] for n in ("q", "k", "v", "do")}
    q, k, v, do = (x[n].to(gpu) for n in ("q", "k", "v", "do"))
    cu_d = torch.tensor(cu, device=gpu)

    def run():
        o, lse = api.forward_varlen(q, k, v, cu_d, max(lens), causal=True)
        return (o, lse) + tuple(api.backward_varlen(q, k, v, o, do, lse, cu_d, max(lens), causal=True))

    o, lse, dq, dk, dv = _reported_then_clean(gpu, run)
    r = ref.attention_varlen(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["do"]), cu, scale=1 / math.sqrt(d),
                             causal=True)
    assert_within({n: compare(n, f64(t), r[n]) for n, t in
                   (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))})


def test_decode_checks_fire_under_slack_and_context_survives(dbg, gpu):
    # 8193 keys: the last key tile starts on the last key row
    B, H, Nq, Nk, d = 2, 3, 1, 8193, 64
    x = workloads.draw(B, H, Nq, d, seed=3, Nk=Nk)
    q, k, v = (x[n].to(gpu) for n in ("q", "k", "v"))

    def run():
        return api.forward_split(q, k, v, causal=True, n_split=4, with_lse=True)

    o, lse = _reported_then_clean(gpu, run)
    r = ref.attention(f64(x["q"]), f64(x["k"]), f64(x["v"]), scale=1 / math.sqrt(d), causal=True, backward=False)
    assert_within({"o": compare("o", f64(o), r["o"]), "lse": compare("lse", f64(lse), r["lse"])})


def test_library_build_is_unaffected(gpu):
    """The library's own build has no debug entry point and still reports a clean word."""
    lib = _lib.load("libfa.so")
    assert not hasattr(lib, "fa_debug_set_check_slack")
    detail = (ctypes.c_int * 4)()
    assert lib.fa_get_last_device_status_detail(ctypes.c_void_p(torch.cuda.current_stream(gpu).cuda_stream),
                                                detail) == 0
