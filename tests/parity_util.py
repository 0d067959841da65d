"""Helpers shared by the GPU parity tests: run the library, run the oracle on
the same bf16 inputs, compare with the stated tolerances."""

import math

import numpy as np
import torch

import workloads
from oracle import ref

# Tolerances: LSE max abs error <= 1e-3; O, dQ, dK, dV max abs error
# <= 2e-2 * max |reference tensor| (bf16 inputs, fp32 accumulation).
LSE_ATOL = 1e-3
REL_TOL = 2e-2
ABS_FLOOR = 1e-4


def run_gpu(x, causal, device, scale=None):
    from io_aware_exact_04_gb300 import api
    q, k, v, do = (x[n].to(device) for n in ("q", "k", "v", "do"))
    kv = None if x["kv_len"] is None else x["kv_len"].to(device)
    o, lse = api.forward(q, k, v, causal=causal, scale=scale, kv_len=kv)
    dq, dk, dv = api.backward(q, k, v, o, do, lse, causal=causal, scale=scale, kv_len=kv)
    torch.cuda.synchronize(device)
    code, detail = api.device_status(device)
    assert code == 0, f"device status {detail}"
    return {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def compare(name, got, want):
    """Max abs error and the bound it must meet."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    if name == "lse":
        ninf = np.isneginf(want)
        assert np.array_equal(ninf, np.isneginf(got)), "LSE -inf pattern differs"
        err = float(np.abs(got[~ninf] - want[~ninf]).max()) if (~ninf).any() else 0.0
        return err, LSE_ATOL
    err = float(np.abs(got - want).max()) if got.size else 0.0
    bound = REL_TOL * float(np.abs(want).max()) if want.size else 0.0
    # Where the mathematics makes the reference tensor identically zero (one
    # valid key: dS = 0, so dQ = dK = 0), the relative bound is 0; fp32
    # accumulation of O(1) bf16 inputs leaves rounding noise of order 1e-6 there.
    return err, max(bound, ABS_FLOOR)


def check_all_heads(B, H, N, d, causal, kv_len=None, seed=0, device=None, qk_scale=1.0, Nk=None):
    """Every head of a [B, H, N, d] problem (keys [B, H, Nk, d]) against the oracle."""
    x = workloads.draw(B, H, N, d, seed=seed, qk_scale=qk_scale,
                       len_range=None, Nk=Nk)
    if kv_len is not None:
        x["kv_len"] = torch.tensor(kv_len, dtype=torch.int32)
    g = run_gpu(x, causal, device)
    r = ref.attention(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["do"]), scale=1 / math.sqrt(d),
                      causal=causal, kv_len=None if kv_len is None else np.asarray(kv_len))
    errs = {}
    for name in ("o", "lse", "dq", "dk", "dv"):
        errs[name] = compare(name, f64(g[name]), r[name])
    return errs


def assert_within(errs):
    bad = {k: v for k, v in errs.items() if not v[0] <= v[1]}
    assert not bad, f"beyond tolerance: {bad} (all: {errs})"
