"""ctypes loader for libgdn.so (the C ABI declared in include/gdn.h).

The library is built in-tree (``chunked_gated_delta_gdn_gb300/_build/libgdn.so``)
by :func:`chunked_gated_delta_gdn_gb300.build.build`.  There is no fallback: if
the library is missing and cannot be built, loading raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

GDN_OK, GDN_ERR_NULL, GDN_ERR_SHAPE, GDN_ERR_DTYPE, GDN_ERR_LAYOUT = 0, 1, 2, 3, 4
GDN_ERR_UNSUPPORTED, GDN_ERR_CUDA, GDN_ERR_WORKSPACE = 5, 6, 7
GDN_F32, GDN_BF16 = 0, 1
GDN_DEV_BAD_SLOT, GDN_DEV_BAD_CU_SEQLENS, GDN_DEV_TIMEOUT = 1, 2, 4

EXPORTS = ("gdn_chunk_fwd", "gdn_chunk_fwd_workspace_size", "gdn_chunk_fwd_path", "gdn_decode",
           "gdn_chunk_fwd_gated", "gdn_decode_gated", "gdn_decode_multi", "gdn_chunk_fwd_noalloc",
           "gdn_product_chunk_fwd", "gdn_product_chunk_fwd_workspace_size", "gdn_product_decode",
           "gdn_chunk_bwd", "gdn_chunk_bwd_workspace_size", "gdn_chunk_bwd_gated",
           "gdn_chunk_bwd_gated_workspace_size", "gdn_selftest_wait_timeout",
           "gdn_status_string", "gdn_version")


class GdnError(RuntimeError):
    """A libgdn entry point returned a status other than GDN_OK."""

    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__("%s failed: %s" % (fn, status_string(status)))


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libgdn.so (building it first when stale and nvcc is available)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if build_if_missing and not _build.up_to_date():
            path = _build.build()
        if not os.path.exists(path):
            raise RuntimeError("libgdn.so not found at %s; run __graft_entry__.build()" % path)
        lib = ctypes.CDLL(path)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.gdn_chunk_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, i, vp, i, vp,
                                      i, vp, i, vp, i, vp, vp, sz, vp, vp]
        lib.gdn_chunk_fwd.restype = i
        lib.gdn_chunk_fwd_workspace_size.argtypes = [i, i, i, i, i, i, i, i, i]
        lib.gdn_chunk_fwd_workspace_size.restype = sz
        lib.gdn_chunk_fwd_path.argtypes = [i, i, i, i]
        lib.gdn_chunk_fwd_path.restype = i
        lib.gdn_decode.argtypes = [vp, vp, vp, vp, vp, vp, i, vp, i, i, i, i, i, i, i, f, i, vp,
                                   vp, vp]
        lib.gdn_decode.restype = i
        lib.gdn_chunk_fwd_gated.argtypes = [vp, vp, vp, vp, vp, i, vp, vp, i, i, i, i, i, i, i,
                                            f, i, vp, i, vp, i, vp, i, vp, i, vp, vp, sz, vp, vp]
        lib.gdn_chunk_fwd_gated.restype = i
        lib.gdn_decode_gated.argtypes = [vp, vp, vp, vp, vp, i, vp, vp, vp, i, vp, i, i, i, i, i,
                                         i, f, i, vp, vp, vp]
        lib.gdn_decode_gated.restype = i
        lib.gdn_decode_multi.argtypes = [vp, vp, vp, vp, vp, vp, i, vp, i, i, i, i, i, i, i, i,
                                         f, i, vp, vp, vp, vp]
        lib.gdn_decode_multi.restype = i
        lib.gdn_product_chunk_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, i, f, i,
                                              vp, i, vp, i, vp, i, vp, i, vp, vp, sz, vp, vp]
        lib.gdn_product_chunk_fwd.restype = i
        lib.gdn_product_chunk_fwd_workspace_size.argtypes = [i, i, i, i, i, i, i, i, i, i]
        lib.gdn_product_chunk_fwd_workspace_size.restype = sz
        lib.gdn_product_decode.argtypes = [vp, vp, vp, vp, vp, vp, i, vp, i, i, i, i, i, i, i, i,
                                           f, i, vp, vp, vp, vp]
        lib.gdn_product_decode.restype = i
        lib.gdn_chunk_bwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, i, vp, i, vp,
                                      i, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp, vp]
        lib.gdn_chunk_bwd.restype = i
        lib.gdn_chunk_bwd_workspace_size.argtypes = [i, i, i, i, i, i, i, i, i]
        lib.gdn_chunk_bwd_workspace_size.restype = sz
        lib.gdn_chunk_bwd_gated.argtypes = [vp, vp, vp, vp, vp, i, vp, vp, i, i, i, i, i, i, i, f,
                                            i, vp, i, vp, i, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                            vp, vp, sz, vp, vp]
        lib.gdn_chunk_bwd_gated.restype = i
        lib.gdn_chunk_bwd_gated_workspace_size.argtypes = [i, i, i, i, i, i, i, i]
        lib.gdn_chunk_bwd_gated_workspace_size.restype = sz
        lib.gdn_selftest_wait_timeout.argtypes = [vp, ctypes.c_ulonglong, i, vp, vp]
        lib.gdn_selftest_wait_timeout.restype = i
        lib.gdn_status_string.argtypes = [i]
        lib.gdn_status_string.restype = ctypes.c_char_p
        lib.gdn_version.argtypes = []
        lib.gdn_version.restype = i
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().gdn_status_string(int(status)).decode()


def check(fn: str, status: int) -> None:
    if status != GDN_OK:
        raise GdnError(fn, status)
