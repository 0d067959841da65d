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
