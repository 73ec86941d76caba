"""ctypes loader for libgqa_attn.so (the C ABI declared in include/gqa_attn.h).

There is no fallback: if the shared library is missing or fails to load, every
call raises.  Build it with ``python -m gqa_head_gated_gb300.build``.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgqa_attn.so")

STATUS = {
    0: "GQA_OK",
    1: "GQA_ERR_INVALID_ARG",
    2: "GQA_ERR_UNSUPPORTED",
    3: "GQA_ERR_CUDA",
    4: "GQA_ERR_TIMEOUT",
    5: "GQA_ERR_WORKSPACE",
    6: "GQA_ERR_DEVICE_RANGE",
}



class LaunchInfo(ctypes.Structure):
    """gqa_launch_info of include/gqa_attn.h."""
    _fields_ = [("kernel", ctypes.c_char * 64), ("seq", ctypes.c_ulonglong),
                ("grid", ctypes.c_uint), ("block", ctypes.c_uint),
                ("dynamic_smem", ctypes.c_uint)]


# name -> (restype, argtypes); the exported symbols of include/gqa_attn.h
_P = ctypes.c_void_p
_I = ctypes.c_int
_FP = ctypes.POINTER(ctypes.c_float)
SIGNATURES = {
    "gqa_status_string": (ctypes.c_char_p, [_I]),
    "gqa_version": (ctypes.c_char_p, []),
    "gqa_attn_prefill": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "gqa_attn_prefill_pair": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "gqa_attn_decode_workspace_size": (ctypes.c_size_t, [_I, _I, _I, _I, _I, _I]),
    "gqa_attn_decode": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P,
                             ctypes.c_size_t, _P]),
    "gqa_attn_decode_plan": (_I, [_I, _I, _I, _I, _I, _I, ctypes.POINTER(_I),
                                  ctypes.POINTER(_I)]),
    "gqa_attn_decode_split": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I,
                                   _I, _P]),
    "attn_lse_merge": (_I, [_P, _P, _I, _I, _P, _P, _P, _P]),
    "gqa_last_device_status": (_I, [_P]),
    "gqa_set_wait_timeout_ns": (None, [ctypes.c_ulonglong]),
    "gqa_selftest_wait_timeout": (_I, [_P, _P]),
    "gqa_kv_append": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P]),
    "gqa_kv_keep": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _P]),
    "gqa_attn_verify_tree": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I,
                                  _P, ctypes.c_size_t, _P]),
    "gqa_attn_decode_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I,
                                     _P]),
    "gqa_launch_log": (_I, [ctypes.POINTER(LaunchInfo), _I]),
    "gqa_attn_mask_check": (_I, [_I, _I, _I, _I, _I, _I, _P, _P, _I]),
    "gqa_attn_masked": (_I, [_P, _P, _P, _P, _P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I,
                             _I, _P]),
}
for _name in ("gqa_attn_masked", "gqa_attn_prefill", "gqa_attn_decode", "gqa_attn_verify_tree",
              "gqa_attn_decode_split", "attn_lse_merge"):
    SIGNATURES[_name + "_f16"] = SIGNATURES[_name]   # fp16 twins, same arguments

_lib = None


class GqaError(RuntimeError):
    def __init__(self, code, where=""):
        self.code = code
        name = STATUS.get(code, str(code))
        super().__init__(f"{where}: {name}" if where else name)


def load():
    """Loads (once) and returns the ctypes handle of libgqa_attn.so."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing; build it with "
                               "`python -m gqa_head_gated_gb300.build`")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def check(code, where=""):
    if code != 0:
        raise GqaError(code, where)
