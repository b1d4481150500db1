"""ctypes declarations of libdflash2's C-ABI (include/dflash2.h).

Loading fails loudly when the library has not been built: there is no other
implementation to fall back to."""
from __future__ import annotations

import ctypes as ct
import os
import re
import threading

from .build import INCLUDE, LIB

_i64, _i32, _int, _vp, _sz, _f32 = ct.c_int64, ct.c_int32, ct.c_int, ct.c_void_p, ct.c_size_t, ct.c_float

SIGNATURES = {
    "dflash2_status_string": (ct.c_char_p, [_int]),
    "dflash2_abi_version": (_int, []),
    "dflash2_kernels_launched": (ct.c_longlong, []),
    "dflash2_unary_topk_path": (_int, [_i64, _i64, _i64, _int]),
    "dflash2_unary_topk_workspace_size": (_sz, [_i64, _i64, _i64, _int, _int]),
    "dflash2_unary_topk": (_int, [_vp, _i64, _i64, _vp, _i64, _int, _f32, _f32, _vp, _int, _vp, _vp, _vp,
                                  _vp, _sz, _vp, _vp]),
    "dflash2_unary_topk_noalloc": (_int, [_vp, _i64, _i64, _vp, _i64, _int, _f32, _f32, _vp, _int, _vp,
                                          _vp, _vp, _vp, _vp]),
    "dflash2_selector_walk": (_int, [_vp, _int, _int, _vp, _vp, _vp, _vp, _vp, _i64, _int, _int, _vp,
                                     _vp, _vp, _vp]),
    "dflash2_selector_pair_scores": (_int, [_vp, _i64, _vp, _vp, _vp, _vp, _vp, _i64, _int, _int,
                                            _vp, _vp, _vp]),
    "dflash2_selector_ce": (_int, [_vp, _vp, _vp, _i64, _int, _i64, _vp, _vp, _vp, _vp]),
    "dflash2_draft_head_workspace_size": (_sz, [_int, _int, _i64, _i64, _int, _int]),
    "dflash2_draft_head": (_int, [_vp, _int, _int, _i64, _vp, _i64, _int, _f32, _f32, _vp, _int, _vp, _vp,
                                  _vp, _vp,
                                  _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp, _vp]),
    "dflash2_selector_lattice": (_int, [_vp, _int, _int, _vp, _vp, _vp, _vp, _vp, _i64, _int, _int,
                                        _vp, _vp, _vp]),
    "dflash2_lattice_walk": (_int, [_vp, _vp, _int, _int, _int, _i64, _vp, ct.c_float, _vp, _vp, _vp,
                                    _vp]),
    "dflash2_conv_prepare_workspace_size": (_sz, [_i64, _int, _int, _int, _int]),
    "dflash2_conv_prepare": (_int, [_vp, _int, _i64, _int, _int, _int, _int, _vp, _vp, _vp, _vp,
                                    _vp, _sz, _vp]),
    "dflash2_selftest_wait_timeout": (_int, [_vp, _i64, _i64, _vp, _i64, _int, _vp, _vp, _vp, _sz, _vp,
                                             _vp]),
    "dflash2_conv_finish": (_int, [_vp, _int, _i64, _int, _int, _int, _int, _vp, _vp, _vp, _vp]),
    "dflash2_conv_finish_prepare_workspace_size": (_sz, [_i64, _int, _int, _int, _int]),
    "dflash2_conv_finish_prepare": (_int, [_vp, _int, _i64, _int, _int, _int, _int, _vp, _vp, _vp, _vp, _vp,
                                           _vp, _vp, _vp, _vp, _sz, _vp]),
}

_lock = threading.Lock()
_lib = None


def header_functions(path: str = os.path.join(INCLUDE, "dflash2.h")) -> list[str]:
    """Names of the functions include/dflash2.h declares."""
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dflash2_[a-z0-9_]+)\s*\(", text)))


def load(path: str = LIB) -> ct.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(
                    f"libdflash2 is not built ({path} missing); run "
                    "`python -m dflash2_draft_block_gb300.build`")
            lib = ct.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
        return _lib
