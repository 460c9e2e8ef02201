"""ctypes declarations of libsfa.so (the C ABI in include/sfa.h).

The library is built in-tree by ``deepseek_sparse_mla_sfa_gb300.build`` into
``deepseek_sparse_mla_sfa_gb300/_build/libsfa.so``.  Loading never falls back to
anything else: a missing or stale library raises.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libsfa.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "sfa.h")

STATUS = {0: "SFA_OK", -1: "SFA_ERR_INVALID_ARG", -2: "SFA_ERR_UNSUPPORTED",
          -3: "SFA_ERR_WORKSPACE", -4: "SFA_ERR_CUDA", -5: "SFA_ERR_DEVICE_TIMEOUT",
          -6: "SFA_ERR_DEVICE_BAD_BLOCK"}

_lock = threading.Lock()
_lib = None

P = ctypes.c_void_p
I = ctypes.c_int
F = ctypes.c_float
SZ = ctypes.c_size_t

SIGNATURES = {
    "sfa_decode": ([P, P, P, P, P, I, I, I, I, I, I, I, F, I, P, P, P, P, P, SZ, P], I),
    "sfa_decode_ex": ([P, P, P, P, P, I, I, I, I, I, I, I, F, I, I, I, P, P, P, P, P, SZ, P], I),
    "sfa_decode_workspace_bytes": ([I, I, I, I, I], SZ),
    "sfa_lse_merge": ([P, P, I, I, I, P, P, P], I),
    "sfa_decode_host_staging_bytes": ([I, I, I, I, I, I], SZ),
    "sfa_decode_host": ([P, P, P, P, P, I, I, I, I, I, I, I, F, I, P, P, P, SZ, P], I),
    "sfa_last_device_status": ([P], I),
    "sfa_status_string": ([I], ctypes.c_char_p),
    "sfa_set_wait_limit": ([ctypes.c_longlong], ctypes.c_longlong),
    "sfa_decode_noalloc": ([P, P, P, P, P, I, I, I, I, I, I, I, F, I, P, P, P], I),
    "sfa_set_kernel_path": ([I], I),
    "sfa_set_stall_injection": ([I], I),
    "sfa_decode_launches": ([I, I, I, I, I, I, I, ctypes.POINTER(ctypes.c_int)], I),
    "sfa_kv_write": ([P, ctypes.c_longlong, P, P, I, P], I),
    "sfa_topk": ([P, ctypes.c_longlong, P, I, I, I, I, P, P], I),
    "sfa_host_plan_create": ([P, P, P, P, P, I, I, I, I, I, I, I, F, I, P, P, P, SZ, P], I),
    "sfa_host_plan_launch": ([P, P], I),
    "sfa_host_plan_destroy": ([P], None),
    "sfa_uv_proj": ([P, P, P, I, I, P], I),
}


class SfaError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {STATUS.get(code, code)}")
        self.code = code


def header_functions(path: str = HEADER):
    """Names of the functions include/sfa.h declares."""
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sfa_[a-z_]+)\s*\(", text)))


def load(path: str = LIB_PATH):
    """Load libsfa.so and declare its signatures (raises if it is missing)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"libsfa.so not found at {path}: build it first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(path)
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def check(fn: str, code: int):
    if code != 0:
        raise SfaError(fn, code)
