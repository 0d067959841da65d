"""tcgen05 operand layouts and the bounded wait, each checked in isolation."""

import ctypes

import pytest
import torch

from io_aware_exact_04_gb300 import _lib

pytestmark = pytest.mark.gpu

A_MN, B_MN, A_TMEM = 1, 2, 4


@pytest.mark.parametrize("mode", [0, A_MN, B_MN, A_MN | B_MN, A_TMEM, A_TMEM | B_MN])
@pytest.mark.parametrize("N,K", [(64, 64), (128, 128), (64, 128), (128, 64)])
def test_tcgen05_gemm_operand_layouts(gpu, mode, N, K):
    g = torch.Generator().manual_seed(N * 1000 + K * 10 + mode)
    # small integers: every product and sum is exact in fp32, so the check is exact
    a = torch.randint(-3, 4, (128, K), generator=g).to(torch.bfloat16)
    b = torch.randint(-3, 4, (K, N), generator=g).to(torch.bfloat16)
    want = a.double() @ b.double()
    a_st = a.t().contiguous() if mode & A_MN else a
    b_st = b if mode & B_MN else b.t().contiguous()
    a_d, b_d = a_st.to(gpu), b_st.to(gpu)
    d = torch.full((128, N), float("nan"), device=gpu)
    status = torch.zeros(4, dtype=torch.int32, device=gpu)
    st = _lib.load("libfa_selftest.so")
    rc = st.fa_selftest_mma(ctypes.c_void_p(a_d.data_ptr()), ctypes.c_void_p(b_d.data_ptr()),
                            ctypes.c_void_p(d.data_ptr()), N, K, mode, ctypes.c_void_p(status.data_ptr()),
                            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    assert status.tolist() == [0, 0, 0, 0]
    assert torch.equal(d.cpu().double(), want)


def test_bounded_wait_gives_up_and_reports(gpu):
    status = torch.zeros(4, dtype=torch.int32, device=gpu)
    st = _lib.load("libfa_selftest.so")
    rc = st.fa_selftest_wait_timeout(ctypes.c_void_p(status.data_ptr()), 20000,
                                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    s = status.tolist()
    assert s[0] == 5 and s[1] == 99  # FA_ERR_TIMEOUT at the self-test's wait site
    # the context is still usable afterwards
    x = torch.ones(1024, device=gpu)
    assert float((x * 2).sum()) == 2048.0
