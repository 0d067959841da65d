"""The allocation-free backward entry point (fa_backward_noalloc).

It serves callers that are handed only input and output buffers and may not
allocate device memory themselves (a runtime that reserves all device memory
up front, say), so the library supplies a fixed scratch array in place of a
workspace. Its gradients must equal those of the workspace entry point
(fa_backward_ex) within the tests' tolerance, call after call, although every
call reuses the same array, and they are checked against the fp64 oracle as
well. This file is collected last so that a stop at the first failure has run
everything else.
"""

import ctypes
import math

import numpy as np
import pytest
import torch

import workloads
from io_aware_exact_04_gb300 import _lib, api
from oracle import ref
from tests.parity_util import assert_within, compare, f64


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def test_rejects_shapes_beyond_the_scratch(built):
    lib = _lib.load("libfa.so")
    cap = lib.fa_backward_noalloc_max_bytes()
    assert cap == 32 << 20
    a = ctypes.c_void_p(0x1000)  # never dereferenced: the size check comes first
    big_n = 1 << 16
    assert lib.fa_backward_workspace_size(1, 16, big_n, 128) > cap
    rc = lib.fa_backward_noalloc(*[a] * 9, 1, 16, big_n, 128, 0.1, 1, None, None)
    assert rc == 2
    assert b"needs" in lib.fa_last_error_detail()
    assert lib.fa_backward_noalloc(*[a] * 9, 1, 1, 128, 96, 0.1, 0, None, None) == 2
    # the common argument checks come first, as in fa_backward_ex: an invalid scale or causal
    # flag on a shape too large for the array is an invalid argument, not an unsupported size
    assert lib.fa_backward_noalloc(*[a] * 9, 1, 16, big_n, 128, 0.0, 1, None, None) == 1
    assert lib.fa_backward_noalloc(*[a] * 9, 1, 16, big_n, 128, 0.1, 2, None, None) == 1
    assert lib.fa_backward_ex(*[a] * 9, 1, 16, big_n, 128, 0.0, 1, None, a, 1 << 40, None) == 1


@pytest.mark.gpu
def test_noalloc_backward_matches_workspace_backward(gpu):
    lib = _lib.load("libfa.so")
    stream = ctypes.c_void_p(torch.cuda.current_stream(gpu).cuda_stream)
    # three calls in a row: a large shape leaves its data in the array, then a smaller shape
    # and another head dimension must not see it, then the first shape again. dK and dV are
    # compared within the tolerance rather than bit for bit: two MMA-issuing warps add into
    # the same dK / dV accumulators in an order that varies between runs, and dQ is a sum of
    # fp32 reduce-adds from many CTAs, so neither entry point repeats its own last bits.
    cases = [(2, 3, 700, 64, True, None), (2, 2, 300, 128, False, [250, 300]), (2, 3, 700, 64, True, None)]
    for B, H, N, d, causal, kv in cases:
        x = workloads.draw(B, H, N, d, seed=N)
        q, k, v, do = (x[n].to(gpu) for n in ("q", "k", "v", "do"))
        kvt = None if kv is None else torch.tensor(kv, dtype=torch.int32, device=gpu)
        scale = 1.0 / math.sqrt(d)
        o, lse = api.forward(q, k, v, causal=causal, kv_len=kvt)
        want = api.backward(q, k, v, o, do, lse, causal=causal, kv_len=kvt)
        got = [torch.full_like(q, float("nan")) for _ in range(3)]
        rc = lib.fa_backward_noalloc(_p(q), _p(k), _p(v), _p(o), _p(do), _p(lse), *(_p(t) for t in got),
                                     B, H, N, d, scale, int(causal), _p(kvt), stream)
        assert rc == 0, lib.fa_last_error_detail()
        torch.cuda.synchronize(gpu)
        assert api.device_status(gpu)[0] == 0
        r = ref.attention(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["do"]), scale=scale, causal=causal,
                          kv_len=None if kv is None else np.asarray(kv))
        errs = {}
        for name, g, w in zip(("dq", "dk", "dv"), got, want):
            gf = g.double().cpu().numpy()
            wf = w.double().cpu().numpy()
            assert np.isfinite(gf).all(), name
            err, bound = compare(name, gf, wf)
            assert err <= bound, (name, err, bound)
            errs[name] = compare(name, gf, r[name])
        assert_within(errs)
