"""The C-ABI library loads, exports what the headers declare, and rejects bad
arguments on the host, before any CUDA call (so these run without a GPU)."""

import ctypes

import pytest

from io_aware_exact_04_gb300 import _lib


@pytest.fixture(scope="module")
def lib(built):
    return _lib.load("libfa.so")


@pytest.mark.parametrize("header,so", [("fa.h", "libfa.so"), ("fa_selftest.h", "libfa_selftest.so")])
def test_exports_every_declared_function(built, header, so):
    names = _lib.declared_functions(header)
    assert len(names) >= 2
    lib = _lib.load(so)
    for name in names:
        assert hasattr(lib, name), name
    assert set(names) == set(_lib.SIGNATURES[so]), "binding signatures and header disagree"


def test_debug_build_exports_the_abi_and_its_own_entry_point(built):
    """libfa_debug.so (bounds-checked build) carries fa.h unchanged plus fa_debug.h; the
    library's own build has no debug entry point."""
    dbg = _lib.load("libfa_debug.so")
    extra = _lib.declared_functions("fa_debug.h")
    assert extra == ["fa_debug_set_check_slack"]
    for name in _lib.declared_functions("fa.h") + extra:
        assert hasattr(dbg, name), name
    assert set(_lib.SIGNATURES["libfa_debug.so"]) == set(extra)
    assert not hasattr(_lib.load("libfa.so"), "fa_debug_set_check_slack")
    # host-side argument check, no CUDA call
    assert dbg.fa_debug_set_check_slack(-1) == 1
    assert dbg.fa_debug_set_check_slack(0) == 0


def test_debug_sites_match_the_header():
    """The site numbers the kernels record are the ones fa_debug.h publishes."""
    import os
    import re
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    with open(os.path.join(root, "include", "fa_debug.h")) as fh:
        header = dict((k, int(v)) for k, v in re.findall(r"(FA_DBG_[A-Z_]+) = (\d+)", fh.read()))
    assert header == {"FA_DBG_META": 100, "FA_DBG_TMA_LOAD": 101, "FA_DBG_TMA_STORE": 102, "FA_DBG_BULK": 103,
                      "FA_DBG_GLOBAL_LOAD": 104, "FA_DBG_GLOBAL_STORE": 105, "FA_DBG_SMEM": 106, "FA_DBG_TMEM": 107}
    with open(os.path.join(root, "io_aware_exact_04_gb300", "csrc", "common.cuh")) as fh:
        aliases = re.findall(r"DBG_([A-Z_]+) = FA_DBG_([A-Z_]+)", fh.read())
    assert len(aliases) == len(header) and all(a == b for a, b in aliases)


def test_status_strings(lib):
    for code in range(7):
        assert lib.fa_status_string(code)
    assert b"unknown" in lib.fa_status_string(99)
    assert lib.fa_version() >= 100


def test_workspace_size_is_linear_in_n(lib):
    def ws(n, d=64):
        return lib.fa_backward_workspace_size(8, 12, n, d)
    assert ws(1024) == 96 * 1024 * (8 + 4 * 64)
    assert ws(2048) == 2 * ws(1024)
    assert ws(1000) == ws(1024)  # padded to 128 rows
    assert lib.fa_backward_workspace_size(2, 16, 4096, 128) == 32 * 4096 * (8 + 4 * 128)
    assert lib.fa_backward_workspace_size(1, 1, 128, 96) == 0


A = ctypes.c_void_p(0x1000)  # 16-byte aligned fake device addresses: never dereferenced
M = ctypes.c_void_p(0x1008)


def fwd(lib, q=A, k=A, v=A, o=A, lse=A, B=1, H=1, N=128, d=64, scale=0.125, causal=0, kv=None):
    return lib.fa_forward_ex(q, k, v, o, lse, B, H, N, d, scale, causal, kv, None)


def bwd(lib, ptrs=None, B=1, H=1, N=128, d=64, scale=0.125, causal=0, ws=A, nbytes=1 << 30):
    p = ptrs or [A] * 9
    return lib.fa_backward_ex(*p, B, H, N, d, scale, causal, None, ws, nbytes, None)


def test_forward_argument_errors(lib):
    assert fwd(lib, d=96) == 2
    assert fwd(lib, d=32) == 2
    assert fwd(lib, causal=2) == 1
    assert fwd(lib, scale=0.0) == 1
    assert fwd(lib, scale=-1.0) == 1
    assert fwd(lib, scale=float("inf")) == 1
    assert fwd(lib, N=-1) == 1
    assert fwd(lib, B=300, H=300) == 2
    assert fwd(lib, q=None) == 1
    assert fwd(lib, lse=None) == 1
    assert fwd(lib, k=M) == 3
    assert fwd(lib, o=M) == 3
    # empty problems are a successful no-op, pointers unused
    assert fwd(lib, q=None, k=None, v=None, o=None, lse=None, N=0) == 0
    assert fwd(lib, q=None, k=None, v=None, o=None, lse=None, B=0) == 0


def test_backward_argument_errors(lib):
    assert bwd(lib, d=96) == 2
    assert bwd(lib, causal=-1) == 1
    assert bwd(lib, ws=None) == 1
    for i in range(9):
        p = [A] * 9
        p[i] = None
        assert bwd(lib, ptrs=p) == 1, i
        p[i] = M
        assert bwd(lib, ptrs=p) == 3, i
    assert bwd(lib, ws=ctypes.c_void_p(0x1010)) == 3  # workspace wants 256-byte alignment
    need = lib.fa_backward_workspace_size(1, 1, 128, 64)
    assert bwd(lib, nbytes=need - 1) == 1
    assert bwd(lib, ptrs=[None] * 9, ws=None, N=0) == 0
    for stage in (-1, 3):
        assert lib.fa_backward_stage(stage, *[A] * 9, 1, 1, 128, 64, 0.125, 0, None, A, 1 << 30, None) == 1
    assert lib.fa_backward_stage(1, *[A] * 9, 1, 1, 128, 96, 0.125, 0, None, A, 1 << 30, None) == 2


def test_unequal_length_argument_errors(lib):
    # queries without keys or keys without queries: unsupported; both empty: nothing to do
    assert lib.fa_forward_qk(*[A] * 5, 1, 1, 0, 5, 64, 0.125, 1, None, None) == 2
    assert lib.fa_forward_qk(*[A] * 5, 1, 1, 5, 0, 64, 0.125, 1, None, None) == 2
    assert lib.fa_forward_qk(*[None] * 5, 1, 1, 0, 0, 64, 0.125, 1, None, None) == 0
    assert lib.fa_forward_qk(*[A] * 5, 1, 1, 5, -1, 64, 0.125, 1, None, None) == 1
    assert lib.fa_backward_qk(*[A] * 9, 1, 1, 0, 7, 64, 0.125, 0, None, A, 1 << 30, None) == 2
    assert lib.fa_backward_qk(*[A] * 9, 1, 1, 3, 7, 96, 0.125, 0, None, A, 1 << 30, None) == 2
    assert lib.fa_backward_stage_qk(3, *[A] * 9, 1, 1, 3, 7, 64, 0.125, 0, None, A, 1 << 30, None) == 1


def test_selftest_argument_errors(built):
    st = _lib.load("libfa_selftest.so")
    assert st.fa_selftest_mma(A, A, A, 96, 64, 0, A, None) == 2
    assert st.fa_selftest_mma(A, A, A, 64, 64, 5, A, None) == 2
    assert st.fa_selftest_mma(None, A, A, 64, 64, 0, A, None) == 1
    assert st.fa_selftest_wait_timeout(None, 10, None) == 1
    assert st.fa_selftest_wait_timeout(A, 0, None) == 1


def test_split_forward_argument_errors(lib):
    need = lib.fa_forward_split_workspace_size(2, 3, 100, 64, 4)
    assert need == ((8 * 6 * 100 * 64 * 4 + 255) // 256) * 256 + ((8 * 6 * 100 * 4 + 255) // 256) * 256
    assert lib.fa_forward_split_workspace_size(2, 3, 100, 96, 4) == 0
    assert lib.fa_forward_split_workspace_size(2, 3, 100, 64, 0) == 0
    args = lambda n_split, ws, nbytes: (*[A] * 5, 2, 3, 100, 900, 64, 0.125, 1, None, n_split, ws, nbytes, None)  # noqa: E731
    W = ctypes.c_void_p(0x10000)
    assert lib.fa_forward_split(*args(0, W, need)) == 1        # no shares
    assert lib.fa_forward_split(*args(2000, W, need)) == 2     # too many shares
    assert lib.fa_forward_split(*args(4, W, need - 1)) == 1    # workspace too small
    assert lib.fa_forward_split(*args(4, None, need)) == 1     # no workspace
    assert lib.fa_forward_split(*args(4, ctypes.c_void_p(0x10010), need)) == 3  # 256-byte alignment
    assert lib.fa_forward_split_count(0, 3, 100, 900, 64) == 1


def test_varlen_argument_errors(lib):
    assert lib.fa_backward_varlen_workspace_size(3, 2, 1000, 64) == (
        2 * (((2 * ((1000 + 12 + 127) // 128 * 128 + 128) * 4) + 255) // 256 * 256) + 2 * 1024 * 64 * 4)
    assert lib.fa_backward_varlen_workspace_size(3, 2, 1000, 96) == 0
    # no cu_seqlens; negative sizes; unsupported head dim
    assert lib.fa_forward_varlen(*[A] * 5, None, 2, 2, 100, 64, 64, 0.125, 0, None) == 1
    assert lib.fa_forward_varlen(*[A] * 6, 2, 2, -1, 64, 64, 0.125, 0, None) == 1
    assert lib.fa_forward_varlen(*[A] * 6, 2, 2, 100, 64, 96, 0.125, 0, None) == 2
    assert lib.fa_forward_varlen(*[None] * 6, 2, 2, 0, 64, 64, 0.125, 0, None) == 0  # nothing to do
    need = lib.fa_backward_varlen_workspace_size(2, 2, 100, 64)
    W = ctypes.c_void_p(0x10000)
    assert lib.fa_backward_varlen(*[A] * 10, 2, 2, 100, 64, 64, 0.125, 0, W, need - 1, None) == 1
    assert lib.fa_backward_varlen(*[A] * 10, 2, 2, 100, 64, 64, 0.125, 0, ctypes.c_void_p(0x10010), need, None) == 3
