"""Parity at the workloads' full sizes, in the launch configuration the
benchmark times: two whole heads compared element by element with the fp64
oracle at every size (up to N = 32768: the oracle works through row blocks of
2048 queries there, exactly), and on every head the invariants that hold at
any size:
  sum_j dK_j = 0            (each row of dS sums to zero)
  sum_j dV_j = sum_i dO_i   (each row of P sums to one; rows with a valid key)
  dK_j = dV_j = 0           for keys beyond the valid length
"""

import pytest
import torch

import workloads
from oracle import ref
from tests.parity_util import assert_within, compare, f64, run_gpu

pytestmark = pytest.mark.gpu

FULL = ["gpt2", "bert", "d128", "long2048", "long8192", "long16384", "long32768", "prefill1024_kv4096"]
INFER = [n for n, w in workloads.WORKLOADS.items() if w.infer]


def _heads(w):
    return [(0, 0), (w.B - 1, w.H - 1)]


@pytest.mark.parametrize("name", FULL)
def test_full_size_whole_head_parity_and_invariants(gpu, name):
    w = workloads.WORKLOADS[name]
    x = workloads.make_inputs(w)
    g = run_gpu(x, w.causal, gpu)
    kv = None if x["kv_len"] is None else x["kv_len"].numpy()

    # ---- oracle on two whole heads
    for b, h in _heads(w):
        q, k, v, do = (f64(x[n][b, h]) for n in ("q", "k", "v", "do"))
        kl = None if kv is None else int(kv[b])
        r = ref.head_backward(q, k, v, do, w.scale, w.causal, kl, row_block=2048 if w.N > 4096 else None)
        errs = {}
        for nm in ("o", "lse", "dq", "dk", "dv"):
            errs[nm] = compare(nm, f64(g[nm][b, h]), r[nm])
        assert_within(errs)

    # ---- invariants on every head (fp64 sums of the bf16 outputs)
    dk = g["dk"].double()
    dv = g["dv"].double()
    dO = x["do"].to(gpu).double()
    sum_dk = dk.sum(dim=2).abs().amax(dim=-1)            # [B, H]
    abs_dk = dk.abs().sum(dim=2).amax(dim=-1)
    assert float((sum_dk / abs_dk).max()) < 2e-3
    if kv is None:
        diff = (dv.sum(dim=2) - dO.sum(dim=2)).abs().amax(dim=-1)
        scale_ = dO.abs().sum(dim=2).amax(dim=-1)
        assert float((diff / scale_).max()) < 2e-3
    else:
        for b in range(w.B):
            n_valid = int(kv[b])
            assert torch.all(g["dk"][b, :, n_valid:] == 0) and torch.all(g["dv"][b, :, n_valid:] == 0)
            diff = (dv[b].sum(dim=1) - dO[b].sum(dim=1)).abs().amax(dim=-1)
            assert float((diff / dO[b].abs().sum(dim=1).amax(dim=-1)).max()) < 2e-3
    lse = g["lse"]
    assert torch.isfinite(lse).all()


@pytest.mark.parametrize("name", INFER)
def test_full_size_inference_forward(gpu, name):
    """The inference workloads at full size, in the bench's launch configuration (the
    library's share count, no LSE), every head against the oracle's forward."""
    from io_aware_exact_04_gb300 import api
    w = workloads.WORKLOADS[name]
    x = workloads.make_inputs(w)
    q, k, v = (x[n].to(gpu) for n in ("q", "k", "v"))
    o, _ = api.forward_split(q, k, v, causal=w.causal)
    o_lse, lse = api.forward_split(q, k, v, causal=w.causal, with_lse=True)
    torch.cuda.synchronize(gpu)
    assert torch.equal(o, o_lse)
    r = ref.attention(f64(x["q"]), f64(x["k"]), f64(x["v"]), scale=w.scale, causal=w.causal, backward=False)
    assert_within({"o": compare("o", f64(o), r["o"]), "lse": compare("lse", f64(lse), r["lse"])})


def test_full_size_packed_sequences():
    """The packed bert workload (16 sequences of 128..512 rows, 16 heads, d 64) at full size, in
    the bench's launch configuration, every (sequence, head) problem against the oracle."""
    from io_aware_exact_04_gb300 import api
    w = workloads.WORKLOADS["bert_packed"]
    x = workloads.make_inputs(w)
    pk = workloads.pack(x)
    lens = x["kv_len"].tolist()
    gpu = torch.device("cuda", 0)
    q, k, v, do = (pk[n].to(gpu) for n in ("q", "k", "v", "do"))
    cu = pk["cu_seqlens"].to(gpu)
    o, lse = api.forward_varlen(q, k, v, cu, max(lens), causal=w.causal)
    dq, dk, dv = api.backward_varlen(q, k, v, o, do, lse, cu, max(lens), causal=w.causal)
    torch.cuda.synchronize(gpu)
    assert api.device_status(gpu)[0] == 0
    r = ref.attention_varlen(f64(pk["q"]), f64(pk["k"]), f64(pk["v"]), f64(pk["do"]), pk["cu_seqlens"].numpy(),
                             scale=w.scale, causal=w.causal)
    assert_within({n: compare(n, f64(t), r[n]) for n, t in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk),
                                                             ("dv", dv))})
