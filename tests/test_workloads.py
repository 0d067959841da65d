"""Seeded workload generator: shapes, determinism, padding lengths, FLOP counts."""

import torch

import workloads


def test_tiny_is_deterministic_and_bf16():
    w = workloads.WORKLOADS["tiny"]
    a = workloads.make_inputs(w)
    b = workloads.make_inputs(w)
    for key in ("q", "k", "v", "do"):
        assert a[key].dtype == torch.bfloat16 and a[key].shape == (1, 1, 128, 64)
        assert torch.equal(a[key], b[key])
    assert a["kv_len"] is None
    # bf16 values are the round-to-nearest of the fp32 draws
    assert torch.equal(a["q"], a["q_f32"].to(torch.bfloat16))


def test_padding_lengths_in_range():
    w = workloads.WORKLOADS["bert"]
    x = workloads.draw(w.B, w.H, 8, 8, len_range=(w.len_lo, w.len_hi))
    kv = x["kv_len"]
    assert kv.dtype == torch.int32 and kv.shape == (w.B,)
    assert int(kv.min()) >= 128 and int(kv.max()) <= 512


def test_qk_scale_applies_to_q_and_k_only():
    a = workloads.draw(1, 1, 16, 8, qk_scale=0.5)
    b = workloads.draw(1, 1, 16, 8)
    assert torch.equal(a["q_f32"], 0.5 * b["q_f32"])
    assert torch.equal(a["k_f32"], 0.5 * b["k_f32"])
    assert torch.equal(a["v_f32"], b["v_f32"])


def test_flop_counts():
    w = workloads.WORKLOADS["gpt2"]
    f = workloads.flop_counts(w)
    # 8*12 heads, 0.5 * 1024^2 * 64 per unit
    unit = 8 * 12 * 0.5 * 1024 * 1024 * 64
    assert f["fwd"] == 4 * unit and f["fwd_bwd_nominal"] == 12 * unit and f["fwd_bwd_executed"] == 14 * unit


def test_visible_pairs_equals_a_half_diagonal_count():
    # brute force: key j of query i counts 1 below the causal bound, 1/2 on it, 0 past it
    import itertools

    def brute(nq, nk, causal, kv):
        tot = 0.0
        for i, j in itertools.product(range(nq), range(min(nk, kv))):
            lim = i + nk - nq
            tot += 1.0 if (not causal or j < lim) else (0.5 if j == lim else 0.0)
        return tot

    for nq, nk, causal, kv in [(4, 4, True, 4), (2, 6, True, 6), (6, 2, True, 2), (4, 6, True, 3),
                               (5, 9, False, 7), (1, 513, True, 513), (700, 300, True, 300),
                               (300, 700, True, 650)]:
        assert abs(workloads.visible_pairs(nq, nk, causal, kv) - brute(nq, nk, causal, kv)) < 1e-9, (nq, nk, kv)
    assert workloads.visible_pairs(1024, 1024, True) == 0.5 * 1024 * 1024


def test_unequal_length_workload_shapes():
    w = workloads.WORKLOADS["prefill1024_kv4096"]
    x = workloads.draw(2, 1, 16, 8, Nk=40)
    assert x["q"].shape == (2, 1, 16, 8) and x["k"].shape == (2, 1, 40, 8) and x["do"].shape == (2, 1, 16, 8)
    assert w.nk == 4096 and w.N == 1024
    f = workloads.flop_counts(w)
    assert f["fwd"] == 4 * 64 * 8 * 12 * (1024 * 4096 - 1024 * 1024 / 2)


def test_pack_keeps_each_sequence_valid_rows_in_order():
    w = workloads.WORKLOADS["bert"]
    x = workloads.draw(4, 3, 40, 8, seed=5, len_range=(3, 40))
    pk = workloads.pack(x)
    kv = x["kv_len"].tolist()
    cu = pk["cu_seqlens"].tolist()
    assert cu[0] == 0 and cu[-1] == sum(kv) and all(b - a == n for a, b, n in zip(cu, cu[1:], kv))
    for name in ("q", "k", "v", "do"):
        assert pk[name].shape == (3, sum(kv), 8) and pk[name].is_contiguous()
        for b in range(4):
            assert torch.equal(pk[name][:, cu[b]:cu[b + 1]], x[name][b, :, :kv[b]])
    assert pk["cu_seqlens"].dtype == torch.int32 and w.packed is False
