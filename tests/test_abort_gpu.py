"""The attention kernels' own abort path: a wait that runs out is reported, not hung.

libfa_withhold.so is a test build of the library in which every CTA leaves out one
of its TMA copies (a flag that nothing sets) and waits give up after 20 ms. Each
kernel must then record FA_ERR_TIMEOUT with a wait site of its own, let its other
copies land, drain its MMAs, free tensor memory and exit; afterwards the context
still runs the normal library correctly. No GPU fault is provoked: every wait in
the kernels is bounded.
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

pytestmark = pytest.mark.gpu

FA_ERR_TIMEOUT = 5
FWD_SITES = range(1, 11)   # the forward kernels' wait sites
BWD_SITES = range(20, 31)  # the backward kernels' wait sites


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


@pytest.fixture(scope="module")
def withhold(gpu):
    return _lib.load("libfa_withhold.so")


def _status(lib, gpu):
    detail = (ctypes.c_int * 4)()
    rc = lib.fa_get_last_device_status_detail(ctypes.c_void_p(torch.cuda.current_stream(gpu).cuda_stream), detail)
    return rc, list(detail)


def _context_still_works(gpu, x, causal):
    """The normal library, on the same context, still matches the oracle."""
    q, k, v, do = (x[n].to(gpu) for n in ("q", "k", "v", "do"))
    o, lse = api.forward(q, k, v, causal=causal)
    dq, dk, dv = api.backward(q, k, v, o, do, lse, causal=causal)
    torch.cuda.synchronize(gpu)
    assert api.device_status(gpu)[0] == 0
    d = q.shape[-1]
    r = ref.attention(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["do"]), scale=1 / math.sqrt(d), causal=causal)
    assert_within({n: compare(n, f64(t), r[n]) for n, t in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))})


# (d, N): the persistent d = 64 forward and the one-CTA-per-item d = 128 forward
@pytest.mark.parametrize("d", [64, 128])
def test_forward_wait_runs_out_and_reports(gpu, withhold, d):
    x = workloads.draw(1, 2, 512, d, seed=d)
    q, k, v = (x[n].to(gpu) for n in ("q", "k", "v"))
    o = torch.full_like(q, float("nan"))
    lse = torch.empty((1, 2, 512), dtype=torch.float32, device=gpu)
    stream = ctypes.c_void_p(torch.cuda.current_stream(gpu).cuda_stream)
    rc = withhold.fa_forward_ex(_p(q), _p(k), _p(v), _p(o), _p(lse), 1, 2, 512, d, 1 / math.sqrt(d), 0, None, stream)
    assert rc == 0
    code, detail = _status(withhold, gpu)
    assert code == FA_ERR_TIMEOUT and detail[0] == FA_ERR_TIMEOUT, detail
    assert detail[1] in FWD_SITES, detail
    assert _status(withhold, gpu)[0] == 0  # reading the word cleared it
    _context_still_works(gpu, x, causal=False)


@pytest.mark.parametrize("d", [64, 128])
def test_backward_wait_runs_out_and_reports(gpu, withhold, d):
    x = workloads.draw(1, 2, 512, d, seed=d + 1)
    q, k, v, do = (x[n].to(gpu) for n in ("q", "k", "v", "do"))
    o, lse = api.forward(q, k, v, causal=True)  # the normal library's forward
    dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
    need = int(withhold.fa_backward_workspace_size(1, 2, 512, d))
    work = torch.empty(need, dtype=torch.uint8, device=gpu)
    stream = ctypes.c_void_p(torch.cuda.current_stream(gpu).cuda_stream)
    rc = withhold.fa_backward_ex(_p(q), _p(k), _p(v), _p(o), _p(do), _p(lse), _p(dq), _p(dk), _p(dv), 1, 2, 512, d,
                                 1 / math.sqrt(d), 1, None, _p(work), need, stream)
    assert rc == 0
    code, detail = _status(withhold, gpu)
    assert code == FA_ERR_TIMEOUT and detail[1] in BWD_SITES, detail
    assert _status(withhold, gpu)[0] == 0
    _context_still_works(gpu, x, causal=True)
