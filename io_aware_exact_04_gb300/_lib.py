"""ctypes binding of the C ABI in include/fa.h (argument marshalling only).

The shared libraries are loaded from this package directory. A missing
library is an ImportError: there is no fallback implementation.
"""

from __future__ import annotations

import ctypes
import os
import re

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)

FA_OK = 0
STATUS_NAMES = {0: "FA_OK", 1: "FA_ERR_INVALID_ARG", 2: "FA_ERR_UNSUPPORTED", 3: "FA_ERR_MISALIGNED",
                4: "FA_ERR_CUDA", 5: "FA_ERR_TIMEOUT", 6: "FA_ERR_DEVICE_CHECK"}

_vp = ctypes.c_void_p
_i = ctypes.c_int
_f = ctypes.c_float
_sz = ctypes.c_size_t

SIGNATURES = {
    "libfa.so": {
        "fa_forward": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp]),
        "fa_forward_ex": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp, _vp]),
        "fa_forward_qk": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _vp, _vp]),
        "fa_backward_varlen": (_i, [_vp] * 10 + [_i, _i, _i, _i, _i, _f, _i, _vp, _sz, _vp]),
        "fa_backward_varlen_workspace_size": (_sz, [_i, _i, _i, _i]),
        "fa_forward_varlen": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _vp]),
        "fa_forward_split": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _vp, _i, _vp, _sz, _vp]),
        "fa_forward_split_workspace_size": (_sz, [_i, _i, _i, _i, _i]),
        "fa_forward_split_count": (_i, [_i, _i, _i, _i, _i]),
        "fa_backward_workspace_size": (_sz, [_i, _i, _i, _i]),
        "fa_backward": (_i, [_vp] * 9 + [_i, _i, _i, _i, _f, _i, _vp, _sz, _vp]),
        "fa_backward_ex": (_i, [_vp] * 9 + [_i, _i, _i, _i, _f, _i, _vp, _vp, _sz, _vp]),
        "fa_backward_stage": (_i, [_i] + [_vp] * 9 + [_i, _i, _i, _i, _f, _i, _vp, _vp, _sz, _vp]),
        "fa_backward_qk": (_i, [_vp] * 9 + [_i, _i, _i, _i, _i, _f, _i, _vp, _vp, _sz, _vp]),
        "fa_backward_stage_qk": (_i, [_i] + [_vp] * 9 + [_i, _i, _i, _i, _i, _f, _i, _vp, _vp, _sz, _vp]),
        "fa_backward_noalloc": (_i, [_vp] * 9 + [_i, _i, _i, _i, _f, _i, _vp, _vp]),
        "fa_backward_noalloc_max_bytes": (_sz, []),
        "fa_status_string": (ctypes.c_char_p, [_i]),
        "fa_get_last_device_status": (_i, [_vp]),
        "fa_get_last_device_status_detail": (_i, [_vp, _vp]),
        "fa_version": (_i, []),
        "fa_last_error_detail": (ctypes.c_char_p, []),
    },
    # builds of the same sources: libfa.so's C ABI plus the entry points listed here
    "libfa_withhold.so": {},  # test build (a withheld copy per CTA)
    "libfa_debug.so": {"fa_debug_set_check_slack": (_i, [_i])},  # include/fa_debug.h
    "libfa_selftest.so": {
        "fa_selftest_mma": (_i, [_vp, _vp, _vp, _i, _i, _i, _vp, _vp]),
        "fa_selftest_wait_timeout": (_i, [_vp, ctypes.c_uint, _vp]),
    },
}

# libraries compiled from the attention sources with other flags
BUILDS_OF_LIBFA = ("libfa_withhold.so", "libfa_debug.so")

_loaded = {}


def lib_path(name: str) -> str:
    return os.path.join(PKG, name)


def load(name: str = "libfa.so") -> ctypes.CDLL:
    if name in _loaded:
        return _loaded[name]
    path = lib_path(name)
    if not os.path.exists(path):
        raise ImportError(f"{path} is not built; run io_aware_exact_04_gb300.build.build()")
    lib = ctypes.CDLL(path)
    sigs = dict(SIGNATURES["libfa.so"]) if name in BUILDS_OF_LIBFA else {}
    sigs.update(SIGNATURES[name])
    for fn, (res, args) in sigs.items():
        f = getattr(lib, fn)
        f.restype = res
        f.argtypes = args
    _loaded[name] = lib
    return lib


def declared_functions(header: str):
    """Names of the functions a public header declares (for export checks)."""
    with open(os.path.join(ROOT, "include", header)) as fh:
        text = fh.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:FA_API\s+)?(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s*(fa_[A-Za-z0-9_]+)\s*\(",
                                 text, flags=re.M)))


class FaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        lib = load()
        msg = lib.fa_status_string(code).decode()
        detail = lib.fa_last_error_detail().decode() if code == 4 else ""
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)} ({msg}){' ' + detail if detail else ''}")


def check(code: int, where: str) -> None:
    if code != FA_OK:
        raise FaError(code, where)
