"""Plain CPU oracle for the float8 training Linear with tensorwise scaling.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package; the library under
``quantised_gemm_gb300`` never does, and it shares no code with it.

The element-wise rules (fp8 codec, amax, scale, cast, delayed update) live in
``fp8_oracle.c``, written scalar from their definitions and compiled with gcc
(-ffp-contract=off, no fast-math).  The GEMM reference is the definition

    y[m, n] = sum_k dec(A[m, k]) * dec(B[n, k]) / (scale_a * scale_b)

evaluated with a library fp64 matrix product (numpy) on operands decoded by
the C codec, plus the absolute sum S[m, n] = sum_k |dec(A) dec(B)| / (s_a s_b)
that the acceptance bound |y - y_ref| <= 2^-7 |y_ref| + 1e-4 S needs.

Sources (page titles):
  * "Integrate float8nocompile, an experimental feature for high performance"
    (pytorch/torchtitan PR 778): Summary (tensorwise dynamic scaling) and the
    single-linear forward+backward benchmark table (ATOMIC_MAX / REDUCTION).
  * "[float8] FP8 GPT 1.5B Delayed Scaling 2x Slower than BF16"
    (pytorch/ao issue 1297): repro script, delayed scaling for input, weight
    and grad_output, enable_amax_init, sync_float8_amax_and_scale_history.
  * "Why swapping nn.Linear with FP8Linear brings throughput decrease for 7B
    LLAMA2-like model?" (pytorch/ao issue 1199): the FP8Linear that replaces
    nn.Linear, i.e. the forward y = x W^T and its two backward products.

Every function is pinned by tests under ``tests/test_oracle_*.py`` (codec
tables against torch's float8 dtypes, closed forms, brute force on tiny
matrices, a hand-worked delayed sequence).  NaN handling is outside the
contract: parity unpinned for NaN inputs.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

E4M3 = 0
E5M2 = 1
FP8_MAX = {E4M3: 448.0, E5M2: 57344.0}
EPS_DEFAULT = 1e-12

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile fp8_oracle.c into oracle/_build/liboracle.so (gcc, OpenMP)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c99", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    c = ctypes
    lib.oracle_fp8_decode.restype = c.c_double
    lib.oracle_fp8_decode.argtypes = [c.c_uint8, c.c_int]
    lib.oracle_fp8_encode.restype = c.c_uint8
    lib.oracle_fp8_encode.argtypes = [c.c_float, c.c_int]
    lib.oracle_fp8_max.restype = c.c_double
    lib.oracle_fp8_max.argtypes = [c.c_int]
    lib.oracle_num_threads.restype = c.c_int
    lib.oracle_amax_bf16.restype = c.c_float
    lib.oracle_amax_bf16.argtypes = [c.c_void_p, c.c_int64, c.c_int64, c.c_int64]
    lib.oracle_scale_dynamic.restype = None
    lib.oracle_scale_dynamic.argtypes = [c.c_float, c.c_float, c.c_int,
                                         c.POINTER(c.c_float), c.POINTER(c.c_float)]
    lib.oracle_scale_delayed.restype = None
    lib.oracle_scale_delayed.argtypes = [c.c_void_p, c.c_int32, c.POINTER(c.c_int32),
                                         c.c_float, c.c_float, c.c_int,
                                         c.POINTER(c.c_float), c.POINTER(c.c_float)]
    lib.oracle_cast_bf16.restype = c.c_float
    lib.oracle_cast_bf16.argtypes = [c.c_void_p, c.c_int64, c.c_int64, c.c_int64,
                                     c.c_float, c.c_int, c.c_void_p, c.c_void_p]
    lib.oracle_encode_f32.restype = None
    lib.oracle_encode_f32.argtypes = [c.c_void_p, c.c_int64, c.c_int, c.c_void_p]
    lib.oracle_decode_array.restype = None
    lib.oracle_decode_array.argtypes = [c.c_void_p, c.c_int64, c.c_int, c.c_void_p]
    lib.oracle_gemm_entries.restype = None
    lib.oracle_gemm_entries.argtypes = [c.c_void_p, c.c_void_p, c.c_int64, c.c_int64,
                                        c.c_int64, c.c_int, c.c_int, c.c_float, c.c_float,
                                        c.c_void_p, c.c_void_p, c.c_int64,
                                        c.c_void_p, c.c_void_p]
    _lib = lib
    return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def num_threads() -> int:
    """OpenMP threads the oracle's loops use."""
    return int(_load().oracle_num_threads())


# ---------------------------------------------------------------- codec

def fp8_max(fmt: int) -> float:
    return float(_load().oracle_fp8_max(fmt))


def decode(code: int, fmt: int) -> float:
    return float(_load().oracle_fp8_decode(code, fmt))


def decode_table(fmt: int) -> np.ndarray:
    """Real value of each of the 256 codes (fp64)."""
    return decode_array(np.arange(256, dtype=np.uint8), fmt)


def decode_array(q: np.ndarray, fmt: int) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.uint8)
    out = np.empty(q.shape, dtype=np.float64)
    _load().oracle_decode_array(_ptr(q), q.size, fmt, _ptr(out))
    return out


def encode(r: float, fmt: int) -> int:
    return int(_load().oracle_fp8_encode(float(r), fmt))


def encode_array(r: np.ndarray, fmt: int) -> np.ndarray:
    """Saturating RNE encode of fp32 values (no scaling)."""
    r = np.ascontiguousarray(r, dtype=np.float32)
    out = np.empty(r.shape, dtype=np.uint8)
    _load().oracle_encode_f32(_ptr(r), r.size, fmt, _ptr(out))
    return out


# ---------------------------------------------------------------- amax / scale

def _as_bf16_bits(x: np.ndarray) -> np.ndarray:
    if x.dtype != np.uint16:
        raise TypeError("oracle takes bf16 tensors as uint16 bit arrays")
    return x


def amax(x: np.ndarray) -> float:
    """max |x| of a 2-D bf16 (uint16 bits) array, as fp32."""
    x = _as_bf16_bits(x)
    if x.ndim != 2:
        raise ValueError("2-D input expected")
    ld = x.strides[0] // 2 if x.shape[0] > 1 else x.shape[1]
    if x.strides[1] != 2:
        x = np.ascontiguousarray(x)
        ld = x.shape[1]
    return float(np.float32(_load().oracle_amax_bf16(_ptr(x), x.shape[0], x.shape[1], ld)))


def scale_dynamic(amax_value: float, fmt: int, eps: float = EPS_DEFAULT):
    """(scale, inv_scale) as fp32: scale = F / max(amax, eps), inv = 1 / scale."""
    s = ctypes.c_float()
    inv = ctypes.c_float()
    _load().oracle_scale_dynamic(float(amax_value), float(eps), fmt,
                                 ctypes.byref(s), ctypes.byref(inv))
    return np.float32(s.value), np.float32(inv.value)


class DelayedState:
    """Delayed scaling state: amax ring of length H, head index, scale.

    Step 0 (amax init): scale comes from the first tensor's own amax and the
    ring is left untouched.  Every step casts with the stored scale; after
    backward ``update(amax_t)`` pushes the step's amax into the ring and
    recomputes the scale from the ring's maximum.
    """

    def __init__(self, history_len: int, fmt: int, eps: float = EPS_DEFAULT):
        if history_len < 1:
            raise ValueError("history length must be >= 1")
        self.H = int(history_len)
        self.fmt = fmt
        self.eps = eps
        self.ring = np.zeros(self.H, dtype=np.float32)
        self.head = 0
        self.scale = None
        self.inv_scale = None

    def init_from(self, amax_value: float):
        self.scale, self.inv_scale = scale_dynamic(amax_value, self.fmt, self.eps)

    def update(self, amax_value: float):
        s = ctypes.c_float()
        inv = ctypes.c_float()
        head = ctypes.c_int32(self.head)
        _load().oracle_scale_delayed(_ptr(self.ring), self.H, ctypes.byref(head),
                                     float(amax_value), float(self.eps), self.fmt,
                                     ctypes.byref(s), ctypes.byref(inv))
        self.head = head.value
        self.scale, self.inv_scale = np.float32(s.value), np.float32(inv.value)


# ---------------------------------------------------------------- cast

def cast(x: np.ndarray, scale: float, fmt: int, transpose: bool = True):
    """(q, qT or None, amax of x): q = sat_rne_fp8(fl32(x * scale))."""
    x = np.ascontiguousarray(_as_bf16_bits(x))
    rows, cols = x.shape
    out = np.empty((rows, cols), dtype=np.uint8)
    out_t = np.empty((cols, rows), dtype=np.uint8) if transpose else None
    a = _load().oracle_cast_bf16(_ptr(x), rows, cols, cols, np.float32(scale), fmt,
                                 _ptr(out), _ptr(out_t) if transpose else None)
    return out, out_t, float(np.float32(a))


def cast_rows(x: np.ndarray, row_idx: np.ndarray, scale: float, fmt: int) -> np.ndarray:
    """Cast only the listed rows of x (for sampled checks at full size)."""
    sub = np.ascontiguousarray(x[row_idx])
    q, _, _ = cast(sub, scale, fmt, transpose=False)
    return q


# ---------------------------------------------------------------- GEMM

def gemm(a8: np.ndarray, b8: np.ndarray, fmt_a: int, fmt_b: int,
         scale_a: float, scale_b: float):
    """(y_ref, S) in fp64 for A [M, K] and B [N, K] (both K fastest)."""
    da = decode_array(a8, fmt_a)
    db = decode_array(b8, fmt_b)
    denom = float(np.float32(scale_a)) * float(np.float32(scale_b))
    y = (da @ db.T) / denom
    s = (np.abs(da) @ np.abs(db).T) / denom
    return y, s


def gemm_entries(a8: np.ndarray, b8: np.ndarray, fmt_a: int, fmt_b: int,
                 scale_a: float, scale_b: float, rows_m: np.ndarray, cols_n: np.ndarray):
    """(y_ref, S) for the listed (m, n) entries only."""
    a8 = np.ascontiguousarray(a8, dtype=np.uint8)
    b8 = np.ascontiguousarray(b8, dtype=np.uint8)
    if a8.shape[1] != b8.shape[1]:
        raise ValueError("contraction lengths differ")
    rm = np.ascontiguousarray(rows_m, dtype=np.int64)
    cn = np.ascontiguousarray(cols_n, dtype=np.int64)
    y = np.empty(rm.size, dtype=np.float64)
    s = np.empty(rm.size, dtype=np.float64)
    K = a8.shape[1]
    _load().oracle_gemm_entries(_ptr(a8), _ptr(b8), K, a8.shape[1], b8.shape[1],
                                fmt_a, fmt_b, np.float32(scale_a), np.float32(scale_b),
                                _ptr(rm), _ptr(cn), rm.size, _ptr(y), _ptr(s))
    return y, s


def gemm_bound(y_ref: np.ndarray, s_ref: np.ndarray) -> np.ndarray:
    """Acceptance bound per entry: 2^-7 |y_ref| + 1e-4 S."""
    return np.ldexp(np.abs(y_ref), -7) + 1e-4 * s_ref


# ---------------------------------------------------------------- Linear step

def linear_fwd_bwd(x, w, dy, scale_x, scale_w, scale_dy):
    """Reference of one forward+backward of the fp8 Linear with given scales.

    Returns dict with the fp8 operands and the fp64 references of
    y = x W^T, dX = dY W and dW = dY^T x on the dequantised operands.
    """
    x8, x8t, _ = cast(x, scale_x, E4M3)
    w8, w8t, _ = cast(w, scale_w, E4M3)
    dy8, dy8t, _ = cast(dy, scale_dy, E5M2)
    y, sy = gemm(x8, w8, E4M3, E4M3, scale_x, scale_w)
    dx, sdx = gemm(dy8, w8t, E5M2, E4M3, scale_dy, scale_w)
    dw, sdw = gemm(dy8t, x8t, E5M2, E4M3, scale_dy, scale_x)
    return dict(x8=x8, x8t=x8t, w8=w8, w8t=w8t, dy8=dy8, dy8t=dy8t,
                y=y, sy=sy, dx=dx, sdx=sdx, dw=dw, sdw=sdw)
