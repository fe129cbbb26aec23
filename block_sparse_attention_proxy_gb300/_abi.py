"""ctypes declarations of the C ABI in include/msa.h (libmsa.so, built in-tree)."""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmsa.so")

MSA_OK = 0
MSA_FLAG_REUSE_REGROUP = 0x1  # msa_bwd: reuse the block lists msa_fwd left in the workspace
MSA_FLAG_TEST_STALL_SELECT = 0x100  # test hook: the selection kernel's first wait runs out
STATUS_NAMES = {
    0: "MSA_OK",
    1: "MSA_ERR_INVALID_ARG",
    2: "MSA_ERR_UNSUPPORTED",
    3: "MSA_ERR_WORKSPACE",
    4: "MSA_ERR_CUDA",
    5: "MSA_ERR_TIMEOUT",
    6: "MSA_ERR_DEVICE_CHECK",
}

# every symbol include/msa.h declares
EXPORTS = (
    "msa_select_workspace_size",
    "msa_fwd_workspace_size",
    "msa_bwd_workspace_size",
    "msa_proxy_select",
    "msa_proxy_select_noalloc",
    "msa_fwd",
    "msa_bwd",
    "msa_get_device_status",
    "msa_last_status_word",
    "msa_launch_count",
    "msa_set_profile_events",
    "msa_status_string",
)


class MsaParams(ctypes.Structure):
    _fields_ = [
        ("total_tokens", ctypes.c_int32),
        ("num_docs", ctypes.c_int32),
        ("max_seqlen", ctypes.c_int32),
        ("hq", ctypes.c_int32),
        ("hkv", ctypes.c_int32),
        ("d", ctypes.c_int32),
        ("dp", ctypes.c_int32),
        ("block", ctypes.c_int32),
        ("top_k", ctypes.c_int32),
        ("window", ctypes.c_int32),
        ("dilation", ctypes.c_int32),
        ("softmax_scale", ctypes.c_float),
        ("proxy_scale", ctypes.c_float),
        ("kl_weight", ctypes.c_float),
        ("flags", ctypes.c_uint32),
    ]


class MsaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")


_lib = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libmsa.so.  Raises if it has not been built: there is no fallback."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build the CUDA library first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    vp, sz, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    P = ctypes.POINTER(MsaParams)
    for name in ("msa_select_workspace_size", "msa_fwd_workspace_size", "msa_bwd_workspace_size"):
        getattr(lib, name).argtypes = [P]
        getattr(lib, name).restype = sz
    lib.msa_proxy_select.argtypes = [P] + [vp] * 8 + [vp, sz, vp]
    lib.msa_proxy_select.restype = i32
    lib.msa_proxy_select_noalloc.argtypes = [P] + [vp] * 8 + [vp]
    lib.msa_proxy_select_noalloc.restype = i32
    lib.msa_fwd.argtypes = [P] + [vp] * 9 + [vp, sz, vp]
    lib.msa_fwd.restype = i32
    lib.msa_bwd.argtypes = [P] + [vp] * 21 + [vp, sz, vp]
    lib.msa_bwd.restype = i32
    lib.msa_get_device_status.argtypes = [vp]
    lib.msa_get_device_status.restype = i32
    lib.msa_last_status_word.argtypes = []
    lib.msa_last_status_word.restype = ctypes.c_uint32
    lib.msa_launch_count.argtypes = []
    lib.msa_launch_count.restype = ctypes.c_uint64
    lib.msa_set_profile_events.argtypes = [i32, vp, vp]
    lib.msa_set_profile_events.restype = i32
    lib.msa_status_string.argtypes = [i32]
    lib.msa_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib
