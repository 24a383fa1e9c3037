"""ctypes declarations of libfp8lin's C ABI (include/fp8lin.h).

Loads ``quantised_gemm_gb300/_build/libfp8lin.so`` (built in-tree by
``quantised_gemm_gb300.build``).  There is no fallback: if the library is
missing or does not load, every call raises.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libfp8lin.so")

# fp8lin_status
OK, EINVAL, EUNSUPPORTED, ECUDA, ETIMEOUT = 0, 1, 2, 3, 4
# fp8lin_fmt
E4M3, E5M2 = 0, 1
# fp8lin_amax_algo
AMAX_ATOMIC, AMAX_REDUCTION, AMAX_SINGLE_PASS, AMAX_AUTO, AMAX_PRECOMPUTED = 0, 1, 2, 3, 4
# fp8lin_scaling
DYNAMIC, DELAYED = 0, 1
# profile kinds
PROF_KINDS = ("amax", "scale", "cast", "cast_fused", "gemm", "small_m")


class ScalingStateC(ctypes.Structure):
    """Mirror of struct fp8lin_scaling_state."""
    _fields_ = [
        ("amax", ctypes.c_void_p),
        ("scale", ctypes.c_void_p),
        ("inv_scale", ctypes.c_void_p),
        ("amax_history", ctypes.c_void_p),
        ("head", ctypes.c_void_p),
        ("history_len", ctypes.c_int32),
        ("fmt", ctypes.c_int32),
        ("kind", ctypes.c_int32),
        ("amax_algo", ctypes.c_int32),
        ("needs_init", ctypes.c_int32),
        ("eps", ctypes.c_float),
    ]


class StepSlotC(ctypes.Structure):
    """Mirror of struct fp8lin_step_slot."""
    _fields_ = [(n, ctypes.c_void_p) for n in ("x", "w", "dy", "y", "dx", "dw", "x8", "x8t", "w8",
                                               "w8t", "dy8", "dy8t", "ws")] + [
        ("ws_bytes", ctypes.c_size_t),
        ("ev", ctypes.c_void_p * 5),
    ]


class Fp8linError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = "%s failed: %s" % (what, status_string(status))
        if status == ECUDA and _lib is not None:
            msg += " (cudaError %d: %s)" % (_lib.fp8lin_last_cuda_error(),
                                            _lib.fp8lin_last_error_detail().decode())
        super().__init__(msg)


_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_SZ = ctypes.c_size_t
_ST = ctypes.POINTER(ScalingStateC)

_SIGNATURES = {
    "fp8lin_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "fp8lin_last_cuda_error": (ctypes.c_int, []),
    "fp8lin_last_error_detail": (ctypes.c_char_p, []),
    "fp8lin_version": (ctypes.c_int, []),
    "fp8lin_workspace_bytes": (_SZ, [_I64, _I64, _I64]),
    "fp8lin_single_pass_max_elems": (_I64, []),
    "fp8lin_check": (ctypes.c_int, [_P, _P]),
    "fp8lin_amax": (ctypes.c_int, [_P, _I64, _I64, _I64, _P, _I32, _P, _P]),
    "fp8lin_amax_noalloc": (ctypes.c_int, [_P, _I64, _I64, _I64, _P, _P]),
    "fp8lin_scale": (ctypes.c_int, [_ST, _P]),
    "fp8lin_scale_many": (ctypes.c_int, [_ST, _I32, _P]),
    "fp8lin_cast": (ctypes.c_int, [_P, _I64, _I64, _I64, _I32, _P, _P, _P, _P, _P]),
    "fp8lin_cast_dynamic": (ctypes.c_int, [_P, _I64, _I64, _I64, _ST, _P, _P, _P, _P]),
    "fp8lin_cast_delayed": (ctypes.c_int, [_P, _I64, _I64, _I64, _ST, _P, _P, _P, _P]),
    "fp8lin_gemm": (ctypes.c_int, [_P, _P, _I64, _I64, _I64, _I64, _I64, _I32, _I32, _P, _P,
                                   _P, _I64, _P, _P, _SZ, _P]),
    "fp8lin_gemm_describe": (ctypes.c_int, [_I64, _I64, _I64, ctypes.c_char_p, _SZ]),
    "fp8lin_gemm_describe_for": (ctypes.c_int,
                                 [_I64, _I64, _I64, ctypes.c_int32, ctypes.c_char_p, _SZ]),
    "fp8lin_gemm_group_describe_for": (ctypes.c_int, [_I64, _I64, _I64, _I64, _I64, _I64,
                                                      ctypes.c_int32, ctypes.c_char_p, _SZ]),
    "fp8lin_forward": (ctypes.c_int, [_P, _P, _I64, _I64, _I64, _ST, _ST, _P, _P, _P, _P, _P,
                                      _P, _P, _SZ, _P]),
    "fp8lin_backward": (ctypes.c_int, [_P, _I64, _I64, _I64, _P, _P, _ST, _ST, _ST, _P, _P,
                                       _P, _P, _P, _P, _P, _SZ, _P]),
    "fp8lin_step_host": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _ST, _ST, _ST,
                                        ctypes.POINTER(StepSlotC), _P, _P, _P, ctypes.c_int]),
    "fp8lin_launch_count": (ctypes.c_uint64, []),
    "fp8lin_profile_enable": (None, [ctypes.c_int]),
    "fp8lin_profile_collect": (ctypes.c_int, [_P, _P]),
    "fp8lin_profile_launches": (_I64, [_P, _P, _I64]),
}


def load(path: str = LIB_PATH):
    """Load libfp8lin (once).  Raises if the shared library is absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            "libfp8lin is not built (%s missing); run __graft_entry__.build() or "
            "python -m quantised_gemm_gb300.build" % path)
    import torch  # noqa: F401  -- loads the CUDA runtime libfp8lin links against
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def status_string(status: int) -> str:
    if _lib is None:
        return "status %d" % status
    return _lib.fp8lin_status_string(status).decode()


def check(status: int, what: str):
    if status != OK:
        raise Fp8linError(status, what)
