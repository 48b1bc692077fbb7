"""ctypes binding of the C ABI in include/moe_fp8_block.h.

Argument marshalling only: every step of the layer runs in the CUDA library.
The library is loaded from this package directory (built in-tree by
build.py); if it is missing, loading raises -- there is no other path.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmoe_fp8_block.so")
ABI_VERSION = 4

MOE_BF16, MOE_F32, MOE_E4M3, MOE_I32 = 1, 2, 3, 4
MOE_PATH_NONE, MOE_PATH_DECODE, MOE_PATH_PREFILL = 0, 1, 2
MOE_STATUS_BAD_ID, MOE_STATUS_TIMEOUT = 1, 2

ERRORS = {
    -1: "MOE_ERR_NULL", -2: "MOE_ERR_DTYPE", -3: "MOE_ERR_SHAPE", -4: "MOE_ERR_ALIGN",
    -5: "MOE_ERR_STRIDE", -6: "MOE_ERR_ALIAS", -7: "MOE_ERR_CAPTURE_GROW", -8: "MOE_ERR_CUDA",
    -9: "MOE_ERR_ARG", -10: "MOE_ERR_DEVICE",
}

# every symbol the header declares
EXPORTS = [
    "moe_fp8_block_forward", "moe_fp8_block_forward_ex", "moe_fp8_block_forward_bias",
    "moe_fp8_block_forward_hostio",
    "moe_fp8_block_forward_decode_noalloc", "moe_fp8_block_noalloc_status", "moe_fp8_block_forward_act_codes",
    "moe_fp8_block_forward_host_experts",
    "moe_fp8_block_route", "moe_fp8_block_act_quant", "moe_fp8_block_widen_e4m3",
    "moe_fp8_block_reserve", "moe_fp8_block_device_status", "moe_fp8_block_last_path", "moe_fp8_block_default_path",
    "moe_fp8_block_last_launches", "moe_fp8_block_set_stage_events", "moe_fp8_block_abi_version", "moe_fp8_block_last_error_detail", "moe_fp8_block_error_string",
    "moe_fp8_block_release",
]


class MoeTensor(ctypes.Structure):
    _fields_ = [
        ("data", ctypes.c_void_p),
        ("ndim", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("shape", ctypes.c_int64 * 4),
        ("stride", ctypes.c_int64 * 4),
    ]


class MoeOptions(ctypes.Structure):
    _fields_ = [
        ("gate_ratio", ctypes.c_float),
        ("force_path", ctypes.c_int32),
        ("decode_act", ctypes.c_int32),
        ("decode_kernel", ctypes.c_int32),
        ("debug_wait_timeout_us", ctypes.c_int32),
        ("debug_drop_stage", ctypes.c_int32),
        ("reserved", ctypes.c_int32 * 2),
    ]


class MoeError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        detail = load().moe_fp8_block_last_error_detail().decode() if code == -8 else ""
        super().__init__(f"{what}: {ERRORS.get(code, code)} ({error_string(code)}) {detail}".rstrip())


_lib = None
_lock = threading.Lock()


def load(path: str = LIB_PATH):
    """Load (once) and return the library; raises if it is missing or stale."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library not built: {path} (run __graft_entry__.build())")
        lib = ctypes.CDLL(path)
        P = ctypes.POINTER
        T = P(MoeTensor)
        i64, i32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
        fwd = [T, T, T, T, T, i64, T, T, i64, T, vp]
        lib.moe_fp8_block_forward.argtypes = fwd
        lib.moe_fp8_block_forward_ex.argtypes = fwd + [P(MoeOptions)]
        lib.moe_fp8_block_forward_hostio.argtypes = fwd + [P(MoeOptions)]
        lib.moe_fp8_block_forward_bias.argtypes = fwd[:9] + [T, T] + fwd[9:] + [P(MoeOptions)]
        lib.moe_fp8_block_forward_decode_noalloc.argtypes = fwd
        lib.moe_fp8_block_forward_act_codes.argtypes = fwd + [P(MoeOptions), vp, vp]
        lib.moe_fp8_block_forward_host_experts.argtypes = fwd + [P(MoeOptions)]
        lib.moe_fp8_block_route.argtypes = [T, i32, vp, vp, vp, vp, vp, vp, vp]
        lib.moe_fp8_block_act_quant.argtypes = [T, vp, vp, vp]
        lib.moe_fp8_block_widen_e4m3.argtypes = [vp, i64, vp, vp]
        lib.moe_fp8_block_reserve.argtypes = [i64, i32, i64, i64, i32, vp]
        lib.moe_fp8_block_device_status.argtypes = [vp, P(ctypes.c_uint32)]
        lib.moe_fp8_block_noalloc_status.argtypes = [vp, P(ctypes.c_uint32)]
        lib.moe_fp8_block_last_path.argtypes = []
        lib.moe_fp8_block_default_path.argtypes = [i64, i32, i32, i64, i64]
        lib.moe_fp8_block_last_launches.argtypes = []
        lib.moe_fp8_block_set_stage_events.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_int]
        lib.moe_fp8_block_abi_version.argtypes = []
        lib.moe_fp8_block_last_error_detail.argtypes = []
        lib.moe_fp8_block_last_error_detail.restype = ctypes.c_char_p
        lib.moe_fp8_block_error_string.argtypes = [ctypes.c_int]
        lib.moe_fp8_block_error_string.restype = ctypes.c_char_p
        lib.moe_fp8_block_release.argtypes = []
        lib.moe_fp8_block_release.restype = None
        v = lib.moe_fp8_block_abi_version()
        if v != ABI_VERSION:
            raise RuntimeError(f"stale CUDA library: ABI {v}, binding expects {ABI_VERSION}")
        _lib = lib
        return lib


def error_string(code: int) -> str:
    lib = load()
    return lib.moe_fp8_block_error_string(code).decode()


def check(rc: int, what: str):
    if rc != 0:
        raise MoeError(rc, what)
