"""The bench's IO accounting (host arithmetic only): compulsory bytes, the standard-attention
N x N term and the step estimate, checked against the terms written out by hand."""

import bench
import workloads


def test_io_accounting_gpt2_terms():
    w = workloads.WORKLOADS["gpt2"]
    heads, N, d = 96, 1024, 64
    io = bench.io_accounting(w, None, measured=100e6)
    fwd = heads * (3 * N * d * 2 + N * d * 2 + N * 4)        # Q, K, V read; O, LSE written
    bwd = heads * (4 * N * d * 2 + N * 4 + 3 * N * d * 2      # Q, K, V, dO, LSE read; dQ, dK, dV written
                   + N * d * 2                                # O read (for D)
                   + 2 * 8 * N + 2 * 4 * N * d)               # -D, -LSE2 and the fp32 accumulator, each written and read
    assert io["compulsory_bytes"] == fwd + bwd
    assert io["standard_attention_bytes"] - io["compulsory_bytes"] == 5 * 2 * heads * N * N
    small = heads * (2 * N * d * 2 + N * 4 + 8 * N + 4 * N * d) + heads * (4 * N * d + 2 * N * d)
    assert io["step_bytes"] == 100e6 + small
    assert abs(io["standard_over_step"] - io["standard_attention_bytes"] / (100e6 + small)) < 1e-12
    assert io["tiled_order_term_bytes"] == heads * 2.0 * N * N * d * d / 116736


def test_io_accounting_counts_only_valid_key_columns():
    w = workloads.WORKLOADS["bert"]
    import torch
    kv = torch.tensor([512] * 8 + [128] * 8, dtype=torch.int32)
    full = bench.io_accounting(w, None)
    part = bench.io_accounting(w, kv)
    assert full["standard_attention_bytes"] - part["standard_attention_bytes"] == 5 * 2 * (8 * 384) * 16 * 512
    assert "step_bytes" not in full  # nothing measured


def test_oracle_units_cover_whole_heads_or_the_last_rows():
    # up to 4096 rows a unit is a whole head; beyond, the last 2048 query rows of each head,
    # whose share of a causal head's pairs is (N^2 - (N - 2048)^2) / 2
    units = bench.oracle_units(workloads.WORKLOADS["gpt2"])
    assert len(units) == 96 and all(r0 == 0 for _, _, r0 in units)
    w = workloads.WORKLOADS["long32768"]
    units = bench.oracle_units(w)
    assert len(units) == 12 and all(r0 == w.N - bench.ORACLE_ROWS for _, _, r0 in units)
    rows = w.N - units[0][2]
    assert workloads.visible_pairs(rows, w.nk, True) == (w.N ** 2 - (w.N - rows) ** 2) / 2


def test_standard_records_pair_the_two_measurements():
    recs = bench.standard_records()
    for wl, rec in recs.items():
        assert rec["standard_attention_dram_bytes"] > rec["flash_step_dram_bytes"] > 0
        assert abs(rec["standard_over_flash"] * rec["flash_step_dram_bytes"]
                   - rec["standard_attention_dram_bytes"]) < 1.0
