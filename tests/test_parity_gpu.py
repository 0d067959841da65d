"""Element-by-element parity of the CUDA path (through the C ABI) with the fp64
oracle, on the same seeded bf16 inputs, plus the degenerate cases."""

import math

import numpy as np
import pytest
import torch

import workloads
from oracle import ref
from tests.parity_util import assert_within, check_all_heads, compare, f64, run_gpu

pytestmark = pytest.mark.gpu

SMALL = [
    # B, H, N, d, causal, kv_len
    (1, 1, 128, 64, False, None),         # the tiny workload's shape: one tile each way
    (1, 2, 384, 64, True, None),          # several tiles, causal diagonal tiles
    (2, 2, 384, 64, False, None),
    (2, 2, 300, 64, False, None),         # ragged tail: 300 = 2*128 + 44
    (2, 2, 300, 64, True, None),
    (1, 1, 700, 64, True, None),          # odd pair count, ragged
    (3, 2, 384, 64, False, [1, 200, 384]),  # key padding incl. a single valid key
    (2, 1, 520, 64, True, [137, 520]),    # causal with key padding
    (1, 2, 256, 128, False, None),        # head dim 128
    (1, 2, 384, 128, True, None),
    (2, 1, 333, 128, True, None),         # head dim 128, ragged
    (2, 2, 200, 128, False, [77, 190]),
    (1, 1, 1, 64, False, None),           # a single row and key
    (1, 1, 1, 128, True, None),
    (1, 1, 17, 64, True, None),
    (1, 2, 1300, 64, True, None),         # d = 64 rows past 1024: the one-CTA-per-item forward grid
    (2, 1, 1100, 64, False, [1100, 3]),
]


@pytest.mark.parametrize("B,H,N,d,causal,kv_len", SMALL)
def test_small_cases_match_oracle(gpu, B, H, N, d, causal, kv_len):
    assert_within(check_all_heads(B, H, N, d, causal, kv_len, seed=N + d, device=gpu))


# The d = 64 backward kernel is persistent: one CTA per SM loops over the key tiles of all
# heads. These shapes give every CTA several tiles (more than 152 tiles), mixing causal and
# full tiles, a ragged last tile, and key padding that leaves whole tiles without a valid key.
MANY_TILES = [
    # B, H, N, d, causal, kv_len
    (8, 24, 256, 64, True, None),                              # 384 tiles
    (6, 20, 300, 64, False, [0, 50, 300, 129, 257, 1]),        # 360 tiles, empty ones included
    (4, 30, 384, 64, True, [384, 200, 10, 384]),               # 360 tiles, causal with padding
    (4, 20, 384, 128, True, [384, 200, 10, 384]),              # d = 128: 240 CTAs, forward in pairs
    (3, 30, 1100, 64, True, [1100, 700, 3]),                   # rows past 1024, forward in pairs, padded
]


@pytest.mark.parametrize("B,H,N,d,causal,kv_len", MANY_TILES)
def test_many_tiles_per_cta_match_oracle(gpu, B, H, N, d, causal, kv_len):
    assert_within(check_all_heads(B, H, N, d, causal, kv_len, seed=7 * N + B, device=gpu))


# Query and key lengths that differ. Causal rows are aligned with the last keys: row i keeps
# keys j <= i + N_k - N_q. Offsets that are not multiples of the 64- or 128-row tiles, more
# queries than keys (leading rows with no key), single queries, and both forward kernels
# (persistent for N_q <= 1024 and N_k <= 1024 at d = 64, one CTA per item otherwise).
UNEQUAL = [
    # B, H, N_q, N_k, d, causal, kv_len
    (2, 3, 128, 1024, 64, True, None),
    (1, 2, 300, 700, 64, True, None),
    (2, 2, 700, 300, 64, True, None),            # rows 0..399 keep no key
    (2, 2, 200, 1500, 64, False, [1500, 37]),
    (1, 3, 1, 513, 64, True, None),
    (1, 2, 64, 3000, 64, True, None),
    (2, 1, 333, 398, 64, True, [398, 100]),      # offset 65
    (1, 2, 600, 129, 64, True, None),            # offset -471
    (1, 2, 256, 640, 128, True, None),
    (2, 1, 384, 200, 128, True, [200, 150]),
    (1, 2, 100, 333, 128, False, None),
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal,kv_len", UNEQUAL)
def test_unequal_query_and_key_lengths_match_oracle(gpu, B, H, Nq, Nk, d, causal, kv_len):
    assert_within(check_all_heads(B, H, Nq, d, causal, kv_len, seed=Nq + 3 * Nk + d, device=gpu, Nk=Nk))


def test_tiny_workload(gpu):
    w = workloads.WORKLOADS["tiny"]
    x = workloads.make_inputs(w)
    g = run_gpu(x, w.causal, gpu)
    r = ref.attention(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["do"]), scale=w.scale, causal=w.causal)
    assert_within({n: compare(n, f64(g[n]), r[n]) for n in ("o", "lse", "dq", "dk", "dv")})


def test_no_valid_key(gpu):
    """kv_len = 0: every score masked; O = 0, LSE = -inf, all gradients zero."""
    errs = check_all_heads(2, 2, 256, 64, False, [0, 256], seed=5, device=gpu)
    assert_within(errs)


def test_empty_sequence_is_noop(gpu):
    from io_aware_exact_04_gb300 import api
    q = torch.empty((2, 3, 0, 64), dtype=torch.bfloat16, device=gpu)
    o, lse = api.forward(q, q, q, causal=True)
    dq, dk, dv = api.backward(q, q, q, o, q, lse, causal=True)
    assert o.shape == q.shape and lse.shape == (2, 3, 0) and dq.shape == q.shape


def test_repeat_runs_are_deterministic(gpu):
    """O and LSE are bitwise repeatable. dQ (fp32 reduce-adds from many CTAs) and,
    at d = 64, dK and dV (two MMA-issuing threads accumulate into them) depend on
    the order of fp32 additions, so repeated runs agree within rounding only."""
    x = workloads.draw(2, 2, 512, 64, seed=3)
    a = run_gpu(x, True, gpu)
    b = run_gpu(x, True, gpu)
    for n in ("o", "lse"):
        assert torch.equal(a[n], b[n]), n
    for n in ("dq", "dk", "dv"):
        diff = (a[n].float() - b[n].float()).abs().max()
        assert diff <= 1e-2 * a[n].float().abs().max(), (n, float(diff))


def test_autograd_function(gpu):
    from io_aware_exact_04_gb300 import api
    x = workloads.draw(1, 2, 256, 64, seed=9)
    q, k, v = (x[n].to(gpu).requires_grad_(True) for n in ("q", "k", "v"))
    o = api.attention(q, k, v, causal=True)
    o.backward(x["do"].to(gpu))
    r = ref.attention(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["do"]), scale=1 / 8, causal=True)
    assert_within({"o": compare("o", f64(o), r["o"]), "dq": compare("dq", f64(q.grad), r["dq"]),
                   "dk": compare("dk", f64(k.grad), r["dk"]), "dv": compare("dv", f64(v.grad), r["dv"])})


# Split-key forward (inference): shares of each item's key tiles joined by a second kernel.
# Uneven shares, more shares than key tiles (empty shares), rows without keys, no LSE.
SPLIT = [
    # B, H, N_q, N_k, d, causal, kv_len, n_split, with_lse
    (1, 2, 1, 4096, 64, True, None, 8, True),
    (2, 3, 128, 3000, 64, True, None, 5, True),
    (2, 2, 300, 2048, 128, False, [2048, 700], 4, True),
    (1, 1, 256, 256, 64, True, None, 3, True),         # 2 key tiles, 3 shares: one is empty
    (3, 1, 64, 1000, 64, False, [1000, 0, 17], 6, True),  # a batch without any valid key
    (2, 2, 16, 5000, 128, True, None, 7, False),
    (1, 2, 1, 700, 64, True, None, 1, False),          # one share, no LSE: still the split path
    # N_q <= 8: the streaming decode kernel. n_split = 1: whole heads a CTA; n_split > 1:
    # min(SMs, 256, n_split B H) CTAs over all heads' key tiles, split heads joined
    (4, 3, 1, 8192, 64, True, None, 8, True),             # heads split between CTAs
    (2, 2, 4, 3000, 128, True, [3000, 1], 5, True),       # causal offset over 4 rows, a one-key batch
    (2, 3, 8, 777, 64, False, [0, 500], 3, False),        # a batch without any valid key
    (1, 1, 3, 100, 64, True, None, 64, True),             # one tile, one CTA
    (3, 2, 2, 1024, 128, False, None, 2, False),
    (2, 3, 2, 1500, 128, True, [1500, 900], 1, True),    # whole heads, padded
    (3, 2, 1, 2000, 64, False, [0, 2000, 129], 1, False),
    (2, 4, 1, 1024, 64, False, None, 1, True),            # one CTA a whole head
    (20, 10, 1, 300, 64, True, None, 1, True),            # more heads than SMs: two whole heads a CTA
    (20, 10, 2, 300, 64, True, [300, 1, 0, 257] * 5, 2, True),  # ... stream-K runs across heads, padded
    (1, 1, 2, 20000, 64, True, None, 64, True),           # one head cut into 64 segments
    (2, 2, 1, 640, 128, False, [0, 0], 2, True),          # no valid key anywhere
    (1, 3, 1, 9000, 128, False, None, 1, True),           # whole heads, d = 128, one query row
    (3, 5, 1, 4000, 128, True, [4000, 2, 3999], 4, True),  # d = 128 key-major lanes, cut heads, padding
    (2, 2, 6, 2500, 128, True, [2500, 1200], 3, True),    # d = 128, up to 8 query rows: cut heads
    (1, 2, 7, 1800, 128, False, None, 1, True),           # ... whole heads
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal,kv_len,n_split,with_lse", SPLIT)
def test_split_key_forward_matches_oracle(gpu, B, H, Nq, Nk, d, causal, kv_len, n_split, with_lse):
    from io_aware_exact_04_gb300 import api
    x = workloads.draw(B, H, Nq, d, seed=Nq + Nk + n_split, Nk=Nk)
    kv = None if kv_len is None else torch.tensor(kv_len, dtype=torch.int32)
    q, k, v = (x[n].to(gpu) for n in ("q", "k", "v"))
    o, lse = api.forward_split(q, k, v, causal=causal, kv_len=None if kv is None else kv.to(gpu),
                               n_split=n_split, with_lse=with_lse)
    torch.cuda.synchronize(gpu)
    code, detail = api.device_status(gpu)
    assert code == 0, f"device status {detail}"
    r = ref.attention(f64(x["q"]), f64(x["k"]), f64(x["v"]), scale=1 / math.sqrt(d), causal=causal,
                      kv_len=None if kv is None else kv.numpy(), backward=False)
    errs = {"o": compare("o", f64(o), r["o"])}
    if with_lse:
        errs["lse"] = compare("lse", f64(lse), r["lse"])
    assert_within(errs)


def test_split_key_forward_default_count_matches_plain_forward(gpu):
    from io_aware_exact_04_gb300 import api
    x = workloads.draw(2, 4, 64, 64, seed=5, Nk=6000)
    q, k, v = (x[n].to(gpu) for n in ("q", "k", "v"))
    o1, lse1 = api.forward(q, k, v, causal=True)
    o2, lse2 = api.forward_split(q, k, v, causal=True, with_lse=True)
    torch.cuda.synchronize(gpu)
    assert float((o1.float() - o2.float()).abs().max()) <= 2e-2 * float(o1.float().abs().max())
    assert float((lse1 - lse2).abs().max()) <= 1e-3


# Packed sequences ([H, T, d], cu_seqlens): ragged lengths, an empty sequence, a single row,
# lengths past one tile pair, both head dims.
VARLEN = [
    # H, lengths, d, causal (d = 64 with every sequence at most 1024 rows runs the persistent
    # forward; longer ones, and d = 128, the one-CTA-per-item forward)
    (2, [100, 0, 257, 643], 64, True),
    (3, [1, 384, 129, 7], 64, False),
    (4, [512, 128, 300, 1, 0, 1024, 77, 256, 640], 64, False),
    (2, [1500, 37, 900], 64, True),
    (2, [300, 1000], 128, True),
    (1, [64, 65, 200, 513], 128, False),
]


def _packed(H, lens, d, seed):
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    x = workloads.draw(1, H, int(cu[-1]), d, seed=seed)
    return cu, {n: x[n][0] for n in ("q", "k", "v", "do")}


@pytest.mark.parametrize("H,lens,d,causal", VARLEN)
def test_packed_sequences_forward_matches_oracle(gpu, H, lens, d, causal):
    from io_aware_exact_04_gb300 import api
    cu, x = _packed(H, lens, d, seed=sum(lens) + d)
    q, k, v = (x[n].to(gpu) for n in ("q", "k", "v"))
    o, lse = api.forward_varlen(q, k, v, torch.tensor(cu, device=gpu), max(lens), causal=causal)
    torch.cuda.synchronize(gpu)
    code, detail = api.device_status(gpu)
    assert code == 0, f"device status {detail}"
    r = ref.attention_varlen(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["do"]), cu, scale=1 / math.sqrt(d),
                             causal=causal, backward=False)
    assert_within({"o": compare("o", f64(o), r["o"]), "lse": compare("lse", f64(lse), r["lse"])})


def test_packed_sequences_longer_than_max_seqlen_are_reported(gpu):
    from io_aware_exact_04_gb300 import api
    cu, x = _packed(1, [100, 300], 64, seed=3)
    q, k, v = (x[n].to(gpu) for n in ("q", "k", "v"))
    api.forward_varlen(q, k, v, torch.tensor(cu, device=gpu), 256, causal=True)  # 300 > 256
    torch.cuda.synchronize(gpu)
    code, detail = api.device_status(gpu)
    assert code == 6, detail  # FA_ERR_DEVICE_CHECK, recorded, no fault


@pytest.mark.parametrize("H,lens,d,causal", VARLEN)
def test_packed_sequences_backward_matches_oracle(gpu, H, lens, d, causal):
    from io_aware_exact_04_gb300 import api
    cu, x = _packed(H, lens, d, seed=2 * sum(lens) + d)
    q, k, v, do = (x[n].to(gpu) for n in ("q", "k", "v", "do"))
    cu_d = torch.tensor(cu, device=gpu)
    o, lse = api.forward_varlen(q, k, v, cu_d, max(lens), causal=causal)
    dq, dk, dv = api.backward_varlen(q, k, v, o, do, lse, cu_d, max(lens), causal=causal)
    torch.cuda.synchronize(gpu)
    code, detail = api.device_status(gpu)
    assert code == 0, f"device status {detail}"
    r = ref.attention_varlen(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["do"]), cu, scale=1 / math.sqrt(d),
                             causal=causal)
    assert_within({n: compare(n, f64(t), r[n]) for n, t in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk),
                                                             ("dv", dv))})
