"""The analytic memory model reproduces every printed cell of the handbook's table."""

import os

import pytest

from io_aware_exact_04_gb300 import memmodel

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [line.split() for line in f if line.strip() and not line.startswith("#")]


@pytest.mark.parametrize("row", _rows("memory_table_gpt2_fp16.txt"))
def test_gpt2_memory_table(row):
    n, std, fl, sav, mat = int(row[0]), float(row[1]), float(row[2]), float(row[3]), float(row[4])
    r = memmodel.training_memory(n, d_model=768, heads=12, layers=12, dtype_bytes=2)
    assert round(r["standard_gb"], 2) == std
    assert round(r["recompute_gb"], 3) == fl
    assert round(r["savings_pct"], 1) == sav
    assert round(r["matrices_gb"], 2) == mat


def test_single_matrix_size():
    (n, b, mb), = _rows("single_attention_matrix.txt")
    nbytes = memmodel.attention_matrix_bytes(int(n), int(b))
    assert nbytes == 134_217_728
    assert round(nbytes / 1e6) == int(mb)


def test_recompute_memory_is_linear_in_n():
    a = memmodel.training_memory(1024, 768, 12, 12)["recompute_bytes"]
    b = memmodel.training_memory(4096, 768, 12, 12)["recompute_bytes"]
    assert b == 4 * a
