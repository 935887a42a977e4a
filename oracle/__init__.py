"""CPU oracle for the NVFP4 batched decode GEMV -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s cpu_baseline /
reference leg may import this package.  The product library never loads it, and
it shares no code with the CUDA path (it builds its own C file with gcc and
talks to it through ctypes).

Every arithmetic step lives in ``nvfp4_oracle.c``; this module only compiles it,
marshals numpy arrays in and out, and adds no arithmetic of its own.

Parity status of each function (pins are in ``tests/test_oracle.py``):
  - e2m1/e4m3/bf16 decode and encode: pinned (spec tables, torch's float8 and
    bfloat16 conversions, exact rational rounding).
  - gemv / gemv_rows / gemv_points: pinned (hand-worked golden cases, brute
    force against a dense numpy float64 reconstruction, invariants).
  - moe_grouped: composition of gemv / gemv_swiglu per routed assignment
    (pinned through them; routing semantics pinned in tests).
  - swiglu / gemv_swiglu: pinned (tabulated sigmoid values, the interleaved
    layout against two separate projections, special cases).
  - quantize: pinned against its definition (hand-derived golden codes, an
    argmin-over-the-code-table restatement, round-trip bounds).  Agreement with
    any third-party NVFP4 quantizer is parity unpinned: the pages print no
    quantized example to check it against.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4_oracle.c")
_LIB = os.path.join(_HERE, "libnvfp4_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C, no FMA contraction, no -march)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
               _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            u8p = ctypes.POINTER(ctypes.c_uint8)
            u16p = ctypes.POINTER(ctypes.c_uint16)
            f32p = ctypes.POINTER(ctypes.c_float)
            f64p = ctypes.POINTER(ctypes.c_double)
            i32p = ctypes.POINTER(ctypes.c_int)
            lib.oracle_e2m1_decode.restype = ctypes.c_double
            lib.oracle_e2m1_decode.argtypes = [ctypes.c_uint]
            lib.oracle_e4m3_decode.restype = ctypes.c_double
            lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint]
            lib.oracle_bf16_decode.restype = ctypes.c_double
            lib.oracle_bf16_decode.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_encode.restype = ctypes.c_uint16
            lib.oracle_bf16_encode.argtypes = [ctypes.c_double]
            lib.oracle_e4m3_encode.restype = ctypes.c_uint
            lib.oracle_e4m3_encode.argtypes = [ctypes.c_double]
            lib.oracle_e2m1_encode.restype = ctypes.c_uint
            lib.oracle_e2m1_encode.argtypes = [ctypes.c_double]
            lib.oracle_quantize.restype = ctypes.c_int
            lib.oracle_quantize.argtypes = [f32p, ctypes.c_int, ctypes.c_int, u8p, u8p, f32p]
            lib.oracle_gemv_rows.restype = ctypes.c_int
            lib.oracle_gemv_rows.argtypes = [u8p, u8p, ctypes.c_float, u16p, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_int, ctypes.c_int, f64p, u16p]
            lib.oracle_gemv_points.restype = ctypes.c_int
            lib.oracle_swiglu.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.c_int, ctypes.c_int,
                                          ctypes.POINTER(ctypes.c_double), u16p]
            lib.oracle_swiglu.restype = ctypes.c_int
            lib.oracle_gemv_points.argtypes = [u8p, u8p, ctypes.c_float, u16p, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int, i32p, i32p, ctypes.c_int, f64p, u16p]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


# ------------------------------------------------------------ scalar codecs
def e2m1_decode(nib: int) -> float:
    return _load().oracle_e2m1_decode(int(nib))


def e4m3_decode(b: int) -> float:
    return _load().oracle_e4m3_decode(int(b))


def bf16_decode(b: int) -> float:
    return _load().oracle_bf16_decode(int(b))


def bf16_encode(v: float) -> int:
    return int(_load().oracle_bf16_encode(float(v)))


def e4m3_encode(v: float) -> int:
    return int(_load().oracle_e4m3_encode(float(v)))


def e2m1_encode(v: float) -> int:
    return int(_load().oracle_e2m1_encode(float(v)))


# ---------------------------------------------------------------- quantizer
def quantize(w: np.ndarray):
    """fp32 W[N, K] -> (packed uint8 [N, K/2], scale uint8 [N, K/16], g float)."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    N, K = w.shape
    packed = np.zeros((N, K // 2), dtype=np.uint8)
    scale = np.zeros((N, K // 16), dtype=np.uint8)
    g = np.zeros(1, dtype=np.float32)
    rc = _load().oracle_quantize(_ptr(w, ctypes.c_float), N, K, _ptr(packed, ctypes.c_uint8),
                                 _ptr(scale, ctypes.c_uint8), _ptr(g, ctypes.c_float))
    if rc != 0:
        raise ValueError(f"oracle_quantize failed with code {rc}")
    return packed, scale, float(g[0])


# --------------------------------------------------------------------- GEMV
def _check_gemv_args(packed, scale, x):
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    scale = np.ascontiguousarray(scale, dtype=np.uint8)
    x = np.ascontiguousarray(x, dtype=np.uint16)
    N, half_k = packed.shape
    K = half_k * 2
    if scale.shape != (N, K // 16) or x.ndim != 2 or x.shape[1] != K:
        raise ValueError("shape mismatch between packed weights, scales and activations")
    return packed, scale, x, N, K


def gemv_rows(packed, scale, g, x, row_begin=0, row_end=None):
    """Y over rows [row_begin, row_end): returns (y64 float64 [n, N], y16 uint16 [n, N]).

    Rows outside the range are left at zero in the returned arrays.
    """
    packed, scale, x, N, K = _check_gemv_args(packed, scale, x)
    n = x.shape[0]
    row_end = N if row_end is None else row_end
    y64 = np.zeros((n, N), dtype=np.float64)
    y16 = np.zeros((n, N), dtype=np.uint16)
    rc = _load().oracle_gemv_rows(_ptr(packed, ctypes.c_uint8), _ptr(scale, ctypes.c_uint8), float(g),
                                  _ptr(x, ctypes.c_uint16), n, N, K, int(row_begin), int(row_end),
                                  _ptr(y64, ctypes.c_double), _ptr(y16, ctypes.c_uint16))
    if rc != 0:
        raise ValueError(f"oracle_gemv_rows failed with code {rc}")
    return y64, y16


def gemv(packed, scale, g, x):
    """Full Y: returns (y64 float64 [n, N], y16 uint16 bf16 bits [n, N])."""
    return gemv_rows(packed, scale, g, x)


def gemv_points(packed, scale, g, x, tok, row):
    """Y at the listed (token, row) pairs: returns (y64 [m], y16 [m])."""
    packed, scale, x, N, K = _check_gemv_args(packed, scale, x)
    n = x.shape[0]
    tok = np.ascontiguousarray(tok, dtype=np.int32)
    row = np.ascontiguousarray(row, dtype=np.int32)
    m = tok.shape[0]
    y64 = np.zeros(m, dtype=np.float64)
    y16 = np.zeros(m, dtype=np.uint16)
    rc = _load().oracle_gemv_points(_ptr(packed, ctypes.c_uint8), _ptr(scale, ctypes.c_uint8), float(g),
                                    _ptr(x, ctypes.c_uint16), n, N, K, _ptr(tok, ctypes.c_int),
                                    _ptr(row, ctypes.c_int), m, _ptr(y64, ctypes.c_double),
                                    _ptr(y16, ctypes.c_uint16))
    if rc != 0:
        raise ValueError(f"oracle_gemv_points failed with code {rc}")
    return y64, y16


# ------------------------------------------------------------------- SwiGLU
def swiglu(gu64):
    """gu64: float64 [n, 2F] (gate/up interleaved columns) -> (h64 [n, F], h16 uint16 bf16 bits [n, F])."""
    gu = np.ascontiguousarray(gu64, dtype=np.float64)
    n, F2 = gu.shape
    F = F2 // 2
    h64 = np.zeros((n, F), dtype=np.float64)
    h16 = np.zeros((n, F), dtype=np.uint16)
    rc = _load().oracle_swiglu(_ptr(gu, ctypes.c_double), n, F, _ptr(h64, ctypes.c_double),
                               _ptr(h16, ctypes.c_uint16))
    if rc != 0:
        raise ValueError(f"oracle_swiglu failed with code {rc}")
    return h64, h16


def gemv_swiglu(packed, scale, g, x):
    """Gate/up projection (rows 2f = gate f, 2f+1 = up f) followed by SwiGLU: (h64, h16) [n, F]."""
    y64, _ = gemv(packed, scale, g, x)
    return swiglu(y64)


# ---------------------------------------------------------- routed experts
def moe_grouped(packed, scale, g, x, expert_offsets, sorted_token, swiglu=False):
    """Per assignment j of expert e (offsets[e] <= j < offsets[e+1]): the expert's
    projection (or gate/up + SwiGLU) of token sorted_token[j].  packed [E][N][K/2],
    scale [E][N][K/16], g [E], x uint16 [n][K].  Returns (y64, y16) [A][N or N/2]."""
    E, N = packed.shape[0], packed.shape[1]
    A = int(expert_offsets[-1])
    width = N // 2 if swiglu else N
    y64 = np.zeros((A, width), dtype=np.float64)
    y16 = np.zeros((A, width), dtype=np.uint16)
    for e in range(E):
        a0, a1 = int(expert_offsets[e]), int(expert_offsets[e + 1])
        if a1 <= a0:
            continue
        xe = np.ascontiguousarray(x[np.asarray(sorted_token[a0:a1], dtype=np.int64)])
        fn = gemv_swiglu if swiglu else gemv
        y64[a0:a1], y16[a0:a1] = fn(packed[e], scale[e], float(g[e]), xe)
    return y64, y16

