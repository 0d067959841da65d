"""Pins of the fp64 oracle against facts fixed by mathematics, not by itself.

Each check would fail for a plausible slip in the oracle: a dropped scale or
term, a wrong sign, a transposed operand, an off-by-one mask. The last group
plants such slips in copies of the oracle's backward and shows the pins catch
them.
"""

import math

import numpy as np
import pytest
import torch

from oracle import ref


def _rand(n, d, seed, scale=1.0):
    r = np.random.default_rng(seed)
    return [scale * r.standard_normal((n, d)) for _ in range(4)]


def _loss(q, k, v, do, s, causal, kv_len):
    o, _ = ref.head_forward(q, k, v, s, causal, kv_len)
    return float((o * do).sum())


def _fd_grad(f, x, h=1e-6):
    g = np.zeros_like(x)
    for idx in np.ndindex(*x.shape):
        old = x[idx]
        x[idx] = old + h
        fp = f()
        x[idx] = old - h
        fm = f()
        x[idx] = old
        g[idx] = (fp - fm) / (2 * h)
    return g


FD_CASES = [
    (1, False, None), (1, True, None),
    (3, False, None), (3, True, None), (3, False, 2),
    (8, False, None), (8, True, None), (8, False, 5), (8, True, 6),
]


def _fd_check(backward_fn, n, causal, kv_len, seed=0):
    d = 4
    q, k, v, do = _rand(n, d, seed)
    s = 1.0 / math.sqrt(d)
    g = backward_fn(q, k, v, do, s, causal, kv_len)
    errs = {}
    for name, x in (("dq", q), ("dk", k), ("dv", v)):
        fd = _fd_grad(lambda: _loss(q, k, v, do, s, causal, kv_len), x)
        denom = max(np.abs(fd).max(), 1e-3)
        errs[name] = np.abs(fd - g[name]).max() / denom
    return errs


@pytest.mark.parametrize("n,causal,kv_len", FD_CASES)
def test_gradients_match_finite_differences(n, causal, kv_len):
    errs = _fd_check(ref.head_backward, n, causal, kv_len)
    for name, e in errs.items():
        assert e < 1e-6, (name, e)


@pytest.mark.parametrize("causal,kv_len", [(False, None), (True, None), (False, 23), (True, 30)])
def test_probability_rows_sum_to_one_and_masked_entries_vanish(causal, kv_len):
    n, d = 37, 8
    q, k, _, _ = _rand(n, d, 1)
    p = ref.probs(q, k, 1 / math.sqrt(d), causal, kv_len)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-12)
    keep = ref.keep_mask(np.arange(n), np.arange(n), causal, kv_len)
    assert np.all(p[~keep] == 0.0)
    assert np.all(p[keep] > 0.0)
    # causal: the diagonal is kept, the first row attends only to key 0
    if causal:
        assert p[0, 0] == 1.0


@pytest.mark.parametrize("causal,kv_len", [(False, None), (True, None), (False, 11)])
def test_rowsum_of_dS_is_zero(causal, kv_len):
    n, d = 29, 8
    q, k, v, do = _rand(n, d, 2)
    it = ref.head_intermediates(q, k, v, do, 1 / math.sqrt(d), causal, kv_len)
    assert np.abs(it["dS"].sum(axis=1)).max() < 1e-12
    # D equals sum_j P_ij dP_ij, the identity behind rowsum(dS) = 0
    np.testing.assert_allclose(it["D"], (it["P"] * it["dP"]).sum(axis=1), atol=1e-12)


def test_single_valid_key_closed_form():
    n, d = 16, 8
    q, k, v, do = _rand(n, d, 3)
    s = 1 / math.sqrt(d)
    g = ref.head_backward(q, k, v, do, s, False, kv_len=1)
    np.testing.assert_allclose(g["o"], np.broadcast_to(v[0], (n, d)), atol=1e-14)
    np.testing.assert_allclose(g["lse"], s * q @ k[0], atol=1e-13)
    np.testing.assert_allclose(g["dv"][0], do.sum(axis=0), atol=1e-12)
    assert np.all(g["dv"][1:] == 0.0)
    assert np.abs(g["dq"]).max() < 1e-12 and np.abs(g["dk"]).max() < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_zero_queries_give_uniform_weights(causal):
    n, d = 20, 8
    _, k, v, do = _rand(n, d, 4)
    q = np.zeros((n, d))
    o, lse = ref.head_forward(q, k, v, 1 / math.sqrt(d), causal)
    if causal:
        cnt = np.arange(1, n + 1)
        np.testing.assert_allclose(o, np.cumsum(v, axis=0) / cnt[:, None], atol=1e-13)
        np.testing.assert_allclose(lse, np.log(cnt), atol=1e-13)
    else:
        np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=0), (n, d)), atol=1e-13)
        np.testing.assert_allclose(lse, np.log(n), atol=1e-13)


def test_causal_first_row():
    n, d = 12, 8
    q, k, v, _ = _rand(n, d, 5)
    s = 1 / math.sqrt(d)
    o, lse = ref.head_forward(q, k, v, s, True)
    np.testing.assert_array_equal(o[0], v[0])
    assert abs(lse[0] - s * q[0] @ k[0]) < 1e-13


def test_fully_masked_rows_are_zero():
    n, d = 10, 8
    q, k, v, do = _rand(n, d, 6)
    g = ref.head_backward(q, k, v, do, 1 / math.sqrt(d), False, kv_len=0)
    assert np.all(g["o"] == 0) and np.all(np.isneginf(g["lse"]))
    for name in ("dq", "dk", "dv"):
        assert np.all(g[name] == 0), name


def _loops_forward(q, k, v, s, causal):
    """Forward by scalar loops and math.exp, for tiny inputs (lists of lists)."""
    n, d = len(q), len(q[0])
    o = [[0.0] * d for _ in range(n)]
    lse = [0.0] * n
    for i in range(n):
        sc = []
        for j in range(n):
            if causal and j > i:
                continue
            sc.append((j, s * sum(q[i][t] * k[j][t] for t in range(d))))
        mx = max(x for _, x in sc)
        den = sum(math.exp(x - mx) for _, x in sc)
        lse[i] = mx + math.log(den)
        for j, x in sc:
            w = math.exp(x - mx) / den
            for t in range(d):
                o[i][t] += w * v[j][t]
    return np.array(o), np.array(lse)


@pytest.mark.parametrize("causal", [False, True])
def test_forward_matches_scalar_loops(causal):
    n, d = 5, 3
    q, k, v, _ = _rand(n, d, 7, scale=2.0)
    o, lse = ref.head_forward(q, k, v, 0.7, causal)
    o2, lse2 = _loops_forward(q.tolist(), k.tolist(), v.tolist(), 0.7, causal)
    np.testing.assert_allclose(o, o2, atol=1e-13)
    np.testing.assert_allclose(lse, lse2, atol=1e-13)


@pytest.mark.parametrize("causal,kv_len", [(False, None), (True, None), (False, 33), (True, 41)])
def test_matches_torch_fp64_autograd(causal, kv_len):
    n, d = 50, 16
    q, k, v, do = _rand(n, d, 8)
    s = 1 / math.sqrt(d)
    g = ref.head_backward(q, k, v, do, s, causal, kv_len)
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    bias = torch.zeros(n, n, dtype=torch.float64)
    i = torch.arange(n)[:, None]
    j = torch.arange(n)[None, :]
    masked = torch.zeros(n, n, dtype=torch.bool)
    if causal:
        masked |= j > i
    if kv_len is not None:
        masked |= j >= kv_len
    bias[masked] = float("-inf")
    logits = (tq @ tk.T) * s + bias
    o = torch.softmax(logits, dim=-1) @ tv
    lse = torch.logsumexp(logits, dim=-1)
    o.backward(torch.tensor(do))
    for name, a, b in (("o", g["o"], o.detach().numpy()), ("lse", g["lse"], lse.detach().numpy()),
                       ("dq", g["dq"], tq.grad.numpy()), ("dk", g["dk"], tk.grad.numpy()),
                       ("dv", g["dv"], tv.grad.numpy())):
        assert np.abs(a - b).max() <= 1e-12 * max(1.0, np.abs(b).max()), name


@pytest.mark.parametrize("causal", [False, True])
def test_large_growing_scores_stay_exact(causal):
    """Scores of several hundred (the regime of the GPU test whose keys' norms ramp up along the
    sequence): the oracle, which subtracts each row's maximum, still matches torch's fp64
    softmax and autograd, and stays finite."""
    n, d = 60, 16
    q, k, v, do = _rand(n, d, 9)
    q = q * 6.0
    k = k * (1.0 + 20.0 * np.arange(n) / n)[:, None]
    s = 1 / math.sqrt(d)
    g = ref.head_backward(q, k, v, do, s, causal)
    assert all(np.isfinite(g[name]).all() for name in ("o", "lse", "dq", "dk", "dv"))
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    logits = (tq @ tk.T) * s
    assert float(logits.detach().abs().max()) > 200.0  # the regime this pins
    if causal:
        logits = logits.masked_fill(torch.ones(n, n, dtype=torch.bool).triu(1), float("-inf"))
    o = torch.softmax(logits, dim=-1) @ tv
    lse = torch.logsumexp(logits, dim=-1)
    o.backward(torch.tensor(do))
    for name, a, b in (("o", g["o"], o.detach().numpy()), ("lse", g["lse"], lse.detach().numpy()),
                       ("dq", g["dq"], tq.grad.numpy()), ("dk", g["dk"], tk.grad.numpy()),
                       ("dv", g["dv"], tv.grad.numpy())):
        assert np.abs(a - b).max() <= 1e-11 * max(1.0, np.abs(b).max()), name


def test_row_groups_do_not_change_results():
    n, d = 300, 16
    q, k, v, do = _rand(n, d, 9)
    s = 1 / math.sqrt(d)
    a = ref.head_backward(q, k, v, do, s, True, None)
    b = ref.head_backward(q, k, v, do, s, True, None, row_block=37)
    for name in a:
        np.testing.assert_allclose(a[name], b[name], rtol=0, atol=1e-12 * max(1.0, np.abs(a[name]).max()))


@pytest.mark.parametrize("causal,kv_len", [(True, None), (False, 250)])
def test_sampled_outputs_match_whole_head(causal, kv_len):
    n, d = 300, 16
    q, k, v, do = _rand(n, d, 10)
    s = 1 / math.sqrt(d)
    full = ref.head_backward(q, k, v, do, s, causal, kv_len)
    rows = [0, 1, 127, 128, 299]
    keys = [0, 5, 200, 260, 299]
    smp = ref.head_sampled(q, k, v, do, s, causal, kv_len, rows, keys, row_block=64)
    for name, idx in (("o", rows), ("lse", rows), ("D", rows), ("dq", rows), ("dk", keys), ("dv", keys)):
        np.testing.assert_allclose(smp[name], full[name][idx], rtol=0, atol=1e-12)


def test_batched_driver_layout_and_head_subset():
    B, H, n, d = 2, 3, 17, 8
    r = np.random.default_rng(11)
    q, k, v, do = (r.standard_normal((B, H, n, d)) for _ in range(4))
    kv = np.array([9, 17])
    allh = ref.attention(q, k, v, do, scale=0.3, causal=False, kv_len=kv)
    assert allh["o"].shape == (B, H, n, d) and allh["lse"].shape == (B, H, n)
    sub = ref.attention(q, k, v, do, scale=0.3, causal=False, kv_len=kv, heads=[(1, 2), (0, 1)])
    np.testing.assert_array_equal(sub["dk"][0], allh["dk"][1, 2])
    np.testing.assert_array_equal(sub["dv"][1], allh["dv"][0, 1])


# ---- planted mistakes: copies of the backward with one slip each ----

def _mutant(kind):
    def bwd(q, k, v, do, s, causal, kv_len):
        n = q.shape[0]
        rows = np.arange(n)
        sm = s * (q @ k.T)
        keep = ref.keep_mask(rows, rows, causal if kind != "diag" else False, kv_len)
        if kind == "diag" and causal:
            keep &= rows[None, :] < rows[:, None]
            keep[0, 0] = True
        sm[~keep] = -np.inf
        p, _, _, _ = ref.softmax_stats(sm)
        o = p @ v
        dd = (do * o).sum(axis=1)
        dv = p.T @ do
        dp = do @ v.T
        ds = p * (dp - (0.0 if kind == "no_D" else dd[:, None]))
        dq = (1.0 if kind == "no_scale" else s) * (ds @ k)
        dk = s * ((ds @ q) if kind == "transpose" else (ds.T @ q))
        if kind == "sign":
            dv = -dv
        return {"dq": dq, "dk": dk, "dv": dv}
    return bwd


@pytest.mark.parametrize("kind", ["no_D", "no_scale", "transpose", "sign", "diag"])
def test_pins_catch_planted_mistakes(kind):
    caught = False
    for n, causal, kv_len in FD_CASES:
        if kind == "diag" and not causal:
            continue
        errs = _fd_check(_mutant(kind), n, causal, kv_len)
        if max(errs.values()) > 1e-3:
            caught = True
            break
    if kind == "diag":
        # an off-by-one causal mask changes the forward itself; the loop pin sees it
        n, d = 5, 3
        q, k, v, _ = _rand(n, d, 7)
        keep = ref.keep_mask(np.arange(n), np.arange(n), False, None) & (np.arange(n)[None, :] < np.arange(n)[:, None])
        keep[0, 0] = True
        sm = 0.7 * (q @ k.T)
        sm[~keep] = -np.inf
        o_bad = ref.softmax_stats(sm)[0] @ v
        o_loop, _ = _loops_forward(q.tolist(), k.tolist(), v.tolist(), 0.7, True)
        caught = caught or np.abs(o_bad - o_loop).max() > 1e-6
    assert caught, kind


# ---- query and key lengths that differ (causal: queries aligned with the last keys) ----

def _rand_qk(nq, nk, d, seed, scale=1.0):
    r = np.random.default_rng(seed)
    return (scale * r.standard_normal((nq, d)), scale * r.standard_normal((nk, d)),
            scale * r.standard_normal((nk, d)), scale * r.standard_normal((nq, d)))


QK_CASES = [  # (N_q, N_k, causal, kv_len)
    (1, 5, True, None), (1, 5, False, None), (5, 2, True, None), (3, 7, False, None),
    (4, 6, True, 4), (6, 3, True, 2), (2, 8, True, 7),
]


@pytest.mark.parametrize("nq,nk,causal,kv_len", QK_CASES)
def test_gradients_match_finite_differences_unequal_lengths(nq, nk, causal, kv_len):
    d = 4
    q, k, v, do = _rand_qk(nq, nk, d, 12)
    s = 1.0 / math.sqrt(d)
    g = ref.head_backward(q, k, v, do, s, causal, kv_len)
    for name, x in (("dq", q), ("dk", k), ("dv", v)):
        fd = _fd_grad(lambda: _loss(q, k, v, do, s, causal, kv_len), x)
        assert np.abs(fd - g[name]).max() / max(np.abs(fd).max(), 1e-3) < 1e-6, name


def _loops_forward_qk(q, k, v, s, causal, kv_len):
    """Scalar loops with the alignment spelled out: query i of N_q is position i + N_k - N_q
    of the key sequence and sees the keys at or before that position."""
    nq, nk, d = len(q), len(k), len(q[0])
    o = [[0.0] * d for _ in range(nq)]
    lse = [-math.inf] * nq
    for i in range(nq):
        pos = i + nk - nq
        sc = [(j, s * sum(q[i][t] * k[j][t] for t in range(d))) for j in range(nk)
              if (not causal or j <= pos) and (kv_len is None or j < kv_len)]
        if not sc:
            continue
        mx = max(x for _, x in sc)
        den = sum(math.exp(x - mx) for _, x in sc)
        lse[i] = mx + math.log(den)
        for j, x in sc:
            for t in range(d):
                o[i][t] += math.exp(x - mx) / den * v[j][t]
    return np.array(o), np.array(lse)


@pytest.mark.parametrize("nq,nk,causal,kv_len", QK_CASES)
def test_forward_matches_scalar_loops_unequal_lengths(nq, nk, causal, kv_len):
    q, k, v, _ = _rand_qk(nq, nk, 3, 13, scale=1.5)
    o, lse = ref.head_forward(q, k, v, 0.6, causal, kv_len)
    o2, lse2 = _loops_forward_qk(q.tolist(), k.tolist(), v.tolist(), 0.6, causal, kv_len)
    np.testing.assert_allclose(o, o2, atol=1e-13)
    np.testing.assert_array_equal(np.isinf(lse), np.isinf(lse2))
    fin = np.isfinite(lse2)
    np.testing.assert_allclose(lse[fin], lse2[fin], atol=1e-13)


def test_fewer_queries_are_the_last_rows_of_the_square_causal_problem():
    # N_q < N_k causal: exactly the last N_q rows of the N_k x N_k causal problem (pinned
    # above by loops, finite differences and torch); with dO zero on the other rows the
    # square problem's dK and dV are those of the short one.
    nq, nk, d = 7, 19, 8
    r = np.random.default_rng(14)
    qf, k, v, dof = (r.standard_normal((nk, d)) for _ in range(4))
    dof[: nk - nq] = 0.0
    s = 0.35
    sq = ref.head_backward(qf, k, v, dof, s, True, None)
    sh = ref.head_backward(qf[nk - nq:], k, v, dof[nk - nq:], s, True, None)
    for name in ("o", "lse", "dq"):
        np.testing.assert_allclose(sh[name], sq[name][nk - nq:], rtol=0, atol=1e-12)
    for name in ("dk", "dv"):
        np.testing.assert_allclose(sh[name], sq[name], rtol=0, atol=1e-12)


def test_more_queries_than_keys_leaves_the_first_rows_empty():
    nq, nk, d = 9, 4, 5
    q, k, v, do = _rand_qk(nq, nk, d, 15)
    g = ref.head_backward(q, k, v, do, 0.4, True, None)
    lead = nq - nk
    assert np.all(g["o"][:lead] == 0) and np.all(np.isneginf(g["lse"][:lead])) and np.all(g["dq"][:lead] == 0)
    sq = ref.head_backward(q[lead:], k, v, do[lead:], 0.4, True, None)  # the square problem
    for name in ("o", "lse", "dq"):
        np.testing.assert_allclose(g[name][lead:], sq[name], rtol=0, atol=1e-12)
    for name in ("dk", "dv"):
        np.testing.assert_allclose(g[name], sq[name], rtol=0, atol=1e-12)


@pytest.mark.parametrize("nq,nk,causal,kv_len", [(20, 45, True, None), (45, 20, True, None),
                                                 (30, 50, False, 33), (24, 40, True, 35)])
def test_matches_torch_fp64_autograd_unequal_lengths(nq, nk, causal, kv_len):
    d = 16
    q, k, v, do = _rand_qk(nq, nk, d, 16)
    s = 1 / math.sqrt(d)
    g = ref.head_backward(q, k, v, do, s, causal, kv_len)
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    pos = torch.arange(nq)[:, None] + (nk - nq)  # each query's position in the key sequence
    j = torch.arange(nk)[None, :]
    masked = torch.zeros(nq, nk, dtype=torch.bool)
    if causal:
        masked |= j > pos
    if kv_len is not None:
        masked |= j >= kv_len
    logits = ((tq @ tk.T) * s).masked_fill(masked, float("-inf"))
    live = ~masked.all(dim=1)  # rows with at least one key; the others are O = 0, LSE = -inf
    p = torch.zeros(nq, nk, dtype=torch.float64)
    p[live] = torch.softmax(logits[live], dim=-1)
    o = p @ tv
    o.backward(torch.tensor(do))
    lse = torch.logsumexp(logits, dim=-1)
    for name, a, b in (("o", g["o"], o.detach().numpy()), ("lse", g["lse"], lse.detach().numpy()),
                       ("dq", g["dq"], tq.grad.numpy()), ("dk", g["dk"], tk.grad.numpy()),
                       ("dv", g["dv"], tv.grad.numpy())):
        fin = np.isfinite(b)
        assert np.array_equal(np.isfinite(a), fin), name
        assert np.abs(a[fin] - b[fin]).max() <= 1e-12 * max(1.0, np.abs(b[fin]).max()), name


def test_pins_catch_a_reversed_alignment():
    # a copy of the mask with the offset's sign flipped (queries aligned with the first keys)
    nq, nk, d = 3, 7, 4
    q, k, v, do = _rand_qk(nq, nk, d, 17)
    sm = 0.5 * (q @ k.T)
    sm[~ref.keep_mask(np.arange(nq), np.arange(nk), True, None, nq - nk)] = -np.inf
    p, _, _, _ = ref.softmax_stats(sm)
    o_bad = p @ v
    o_loop, _ = _loops_forward_qk(q.tolist(), k.tolist(), v.tolist(), 0.5, True, None)
    assert np.abs(o_bad - o_loop).max() > 1e-3


# ---- packed sequences (each sequence its own problem) ----

@pytest.mark.parametrize("causal", [False, True])
def test_packed_sequences_equal_the_padded_batch_with_key_padding(causal):
    # the same numbers through the mask route: a padded [B, H, Lmax, d] batch with key padding
    # kv_len = len_b and dO zero on the padding rows (so they add nothing to dK, dV)
    lens, H, d = [5, 9, 1, 0, 7], 2, 4
    cu = np.concatenate([[0], np.cumsum(lens)])
    T, L = int(cu[-1]), max(lens)
    r = np.random.default_rng(18)
    q, k, v, do = (r.standard_normal((H, T, d)) for _ in range(4))
    s = 0.45
    got = ref.attention_varlen(q, k, v, do, cu, scale=s, causal=causal)
    B = len(lens)
    pad = lambda x: np.stack([np.pad(x[:, cu[b]:cu[b + 1]], ((0, 0), (0, L - lens[b]), (0, 0))) for b in range(B)])  # noqa: E731
    want = ref.attention(pad(q), pad(k), pad(v), pad(do), scale=s, causal=causal, kv_len=np.array(lens))
    for b in range(B):
        for name in ("o", "dq", "dk", "dv"):
            np.testing.assert_allclose(got[name][:, cu[b]:cu[b + 1]], want[name][b, :, :lens[b]], rtol=0, atol=1e-12)
        np.testing.assert_allclose(got["lse"][:, cu[b]:cu[b + 1]], want["lse"][b, :, :lens[b]], rtol=0, atol=1e-12)


def test_packed_sequences_do_not_see_each_other():
    H, d = 1, 4
    r = np.random.default_rng(19)
    q, k, v, do = (r.standard_normal((H, 12, d)) for _ in range(4))
    two = ref.attention_varlen(q, k, v, do, [0, 6, 12], scale=0.5, causal=False)
    one = ref.attention_varlen(q, k, v, do, [0, 12], scale=0.5, causal=False)
    assert np.abs(two["o"][:, 6:] - one["o"][:, 6:]).max() > 1e-3
    solo = ref.head_forward(q[0, 6:], k[0, 6:], v[0, 6:], 0.5, False)[0]
    np.testing.assert_allclose(two["o"][0, 6:], solo, rtol=0, atol=1e-12)
