"""ctypes front end of the CPU oracle (oracle.c).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module; the product library
never does.  It compiles ``oracle.c`` with gcc on first use (or when
``build()`` is called) into ``oracle/_build/liboracle.so``.

Arrays are numpy: bf16 activations travel as ``uint16`` bit patterns, Q4_K
weights as ``uint8`` byte arrays of shape ``[rows, ceil(cols/256) * 144]``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

QK = 256
QK_BYTES = 144

# block formats of W_down (the values match the library's format codes only by
# the shared reading of the pages; nothing is imported from it)
FMT_Q4_K, FMT_Q5_K, FMT_Q6_K, FMT_Q5_1 = 0, 1, 2, 3
_FMT_BLOCK = {FMT_Q4_K: (256, 144), FMT_Q5_K: (256, 176), FMT_Q6_K: (256, 210), FMT_Q5_1: (32, 24)}


def row_bytes_fmt(fmt: int, cols: int) -> int:
    bw, bb = _FMT_BLOCK[fmt]
    return ((cols + bw - 1) // bw) * bb


def row_bytes(cols: int) -> int:
    return ((cols + QK - 1) // QK) * QK_BYTES


_FLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile oracle.c (plain C, -O2, no fast-math, no FMA contraction,
    single-threaded: its OpenMP pragmas are ignored)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", *_FLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_OMP_PATH = os.path.join(_OUT_DIR, "liboracle_omp.so")


def build_omp(force: bool = False):
    """The same source built with -fopenmp: its independent row loops run on
    all host cores (the CPU baseline's all-cores leg).  Returns the library
    path, or None where the compiler has no OpenMP."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    stale = (not os.path.exists(_OMP_PATH)
             or os.path.getmtime(_OMP_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _OMP_PATH + f".{os.getpid()}.tmp"
        try:
            subprocess.check_call(["gcc", *_FLAGS, "-fopenmp", "-o", tmp, _SRC, "-lm"],
                                  stderr=subprocess.DEVNULL)
        except (subprocess.CalledProcessError, OSError):
            return None
        os.replace(tmp, _OMP_PATH)
    return _OMP_PATH


def use_library(path: str):
    """Route the wrappers to another build of oracle.c (e.g. build_omp());
    returns the previous path, for restoring."""
    global _lib, _active
    with _lock:
        prev = _active
        _active = path
        _lib = None
    return prev


_active = None


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(_active or build())
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            lib.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
            lib.oracle_f16_to_f32.restype = ctypes.c_float
            lib.oracle_f32_to_f16.argtypes = [ctypes.c_float]
            lib.oracle_f32_to_f16.restype = ctypes.c_uint16
            lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_f32.restype = ctypes.c_float
            lib.oracle_silu.argtypes = [ctypes.c_double]
            lib.oracle_silu.restype = ctypes.c_double
            lib.oracle_q4k_scale_min.argtypes = [P, ctypes.c_int, P, P]
            lib.oracle_q4k_dequant.argtypes = [P, P, I64, I64]
            lib.oracle_q4k_quantize.argtypes = [P, P, I64, I64]
            lib.oracle_swiglu_ffn.argtypes = [P, P, P, P, I64, I64, I64, P]
            lib.oracle_moe_swiglu_ffn.argtypes = [P, P, P, P, P, P, I64, I64, I64, I64, I64, P]
            lib.oracle_route_top_k.argtypes = [P, I64, I64, I64, P, P]
            lib.oracle_dequant_fmt.argtypes = [ctypes.c_int, P, P, I64, I64]
            lib.oracle_swiglu_ffn_fmt.argtypes = [P, P, P, P, ctypes.c_int, I64, I64, I64, P]
            lib.oracle_moe_swiglu_ffn_fmt.argtypes = [P, P, P, P, P, P, ctypes.c_int, I64, I64, I64,
                                                      I64, I64, P]
            lib.oracle_moe_swiglu_ffn_scaled.argtypes = [P, P, P, P, P, P, P, ctypes.c_int, I64, I64,
                                                         I64, I64, I64, P]
            lib.oracle_fmt_row_bytes.argtypes = [ctypes.c_int, I64]
            lib.oracle_fmt_row_bytes.restype = I64
            lib.oracle_bf16_from_f64.argtypes = [ctypes.c_double]
            lib.oracle_bf16_from_f64.restype = ctypes.c_uint16
            lib.oracle_rmsnorm_bf16.argtypes = [P, P, ctypes.c_double, I64, I64, P]
            for f in ("oracle_q4k_dequant", "oracle_q4k_quantize",
                      "oracle_swiglu_ffn", "oracle_moe_swiglu_ffn",
                      "oracle_q4k_scale_min"):
                getattr(lib, f).restype = None
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


# ---- scalar helpers ------------------------------------------------------

def f16_to_f32(bits: int) -> float:
    return float(_load().oracle_f16_to_f32(int(bits)))


def f32_to_f16(x: float) -> int:
    return int(_load().oracle_f32_to_f16(float(x)))


def bf16_to_f32(bits: int) -> float:
    return float(_load().oracle_bf16_to_f32(int(bits)))


def silu(g: float) -> float:
    return float(_load().oracle_silu(float(g)))


def scale_min(scales12: bytes, j: int):
    buf = np.frombuffer(bytes(scales12), dtype=np.uint8).copy()
    sc = ctypes.c_int()
    m = ctypes.c_int()
    _load().oracle_q4k_scale_min(_ptr(buf), int(j), ctypes.byref(sc), ctypes.byref(m))
    return sc.value, m.value


# ---- Q4_K ----------------------------------------------------------------

def q4k_dequant(blocks: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """Dequantise ``rows`` rows of Q4_K blocks to an fp32 [rows, cols] array."""
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
    assert blocks.size >= rows * row_bytes(cols)
    out = np.empty((rows, cols), dtype=np.float32)
    _load().oracle_q4k_dequant(_ptr(blocks), _ptr(out), rows, cols)
    return out


def q4k_quantize(w: np.ndarray) -> np.ndarray:
    """Quantise an fp32 [rows, cols] matrix to Q4_K rows (min/max quantiser)."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    rows, cols = w.shape
    out = np.zeros((rows, row_bytes(cols)), dtype=np.uint8)
    _load().oracle_q4k_quantize(_ptr(w), _ptr(out), rows, cols)
    return out


# ---- feed-forward ----------------------------------------------------------

def swiglu_ffn(x_bf16: np.ndarray, Wg: np.ndarray, Wu: np.ndarray, Wd: np.ndarray,
               T: int, H: int, I: int, wd_fmt: int = FMT_Q4_K) -> np.ndarray:
    """y[T, H] in float64 for bf16 bits x[T, H], Q4_K W_gate and W_up, and W_down
    in block format wd_fmt."""
    x_bf16 = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    Wg = np.ascontiguousarray(Wg, dtype=np.uint8)
    Wu = np.ascontiguousarray(Wu, dtype=np.uint8)
    Wd = np.ascontiguousarray(Wd, dtype=np.uint8)
    assert x_bf16.size == T * H
    assert Wg.size == I * row_bytes(H) and Wu.size == I * row_bytes(H)
    assert Wd.size == H * row_bytes_fmt(wd_fmt, I)
    y = np.empty((T, H), dtype=np.float64)
    _load().oracle_swiglu_ffn_fmt(_ptr(x_bf16), _ptr(Wg), _ptr(Wu), _ptr(Wd), wd_fmt, T, H, I,
                                  _ptr(y))
    return y


def moe_swiglu_ffn(x_bf16: np.ndarray, ids: np.ndarray, wts: np.ndarray,
                   Wg: np.ndarray, Wu: np.ndarray, Wd: np.ndarray,
                   T: int, H: int, I: int, E: int, top_k: int,
                   wd_fmt: int = FMT_Q4_K, down_scale=None) -> np.ndarray:
    """y[T, H] float64 for the routed experts; weights stacked [E, rows, bytes],
    W_down in block format wd_fmt; down_scale: None or fp32 [E], a scale on
    each expert's down projection."""
    x_bf16 = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    wts = np.ascontiguousarray(wts, dtype=np.float32)
    Wg = np.ascontiguousarray(Wg, dtype=np.uint8)
    Wu = np.ascontiguousarray(Wu, dtype=np.uint8)
    Wd = np.ascontiguousarray(Wd, dtype=np.uint8)
    assert ids.size == T * top_k and wts.size == T * top_k
    assert Wg.size == E * I * row_bytes(H) and Wd.size == E * H * row_bytes_fmt(wd_fmt, I)
    y = np.empty((T, H), dtype=np.float64)
    if down_scale is None:
        sc = None
    else:
        down_scale = np.ascontiguousarray(down_scale, dtype=np.float32)
        assert down_scale.size == E
        sc = _ptr(down_scale)
    _load().oracle_moe_swiglu_ffn_scaled(_ptr(x_bf16), _ptr(ids), _ptr(wts), sc, _ptr(Wg), _ptr(Wu),
                                         _ptr(Wd), wd_fmt, T, H, I, E, top_k, _ptr(y))
    return y


def dequant_fmt(blocks: np.ndarray, fmt: int, rows: int, cols: int) -> np.ndarray:
    """fp32 [rows, cols] from rows of blocks of format fmt."""
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
    assert blocks.size == rows * row_bytes_fmt(fmt, cols)
    out = np.empty((rows, cols), dtype=np.float32)
    _load().oracle_dequant_fmt(fmt, _ptr(blocks), _ptr(out), rows, cols)
    return out


def route_top_k(logits: np.ndarray, top_k: int):
    """(ids int32 [T, top_k], weights float32 [T, top_k]) for logits [T, E].

    The top_k experts of each token from the highest logit down (ties to the
    lower index, NaN below every number), with softmax weights over the chosen
    logits, evaluated in fp64 and rounded once to fp32."""
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = logits.shape
    assert 1 <= top_k <= E
    ids = np.empty((T, top_k), dtype=np.int32)
    w = np.empty((T, top_k), dtype=np.float32)
    _load().oracle_route_top_k(_ptr(logits), T, E, top_k, _ptr(ids), _ptr(w))
    return ids, w


def bf16_from_f64(v: float) -> int:
    """bf16 bits of v rounded once to nearest even (normal range)."""
    return int(_load().oracle_bf16_from_f64(float(v)))


def rmsnorm_bf16(h: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """bf16 bits (uint16 [T, H]) of h / sqrt(mean(h^2) + eps) * gamma per row."""
    h = np.ascontiguousarray(h, dtype=np.float32)
    gamma = np.ascontiguousarray(gamma, dtype=np.float32)
    T, H = h.shape
    assert gamma.shape == (H,)
    x = np.empty((T, H), dtype=np.uint16)
    _load().oracle_rmsnorm_bf16(_ptr(h), _ptr(gamma), float(eps), T, H, _ptr(x))
    return x


def prenorm_swiglu_residual(h: np.ndarray, gamma: np.ndarray, eps: float, Wg: np.ndarray,
                            Wu: np.ndarray, Wd: np.ndarray, I: int):
    """(h + block(x), x) with x = rmsnorm_bf16(h, gamma, eps): the block with
    its normalisation and residual connection; float64 [T, H] and bf16 bits."""
    T, H = h.shape
    x = rmsnorm_bf16(h, gamma, eps)
    y = swiglu_ffn(x, Wg, Wu, Wd, T, H, I)
    return np.asarray(h, dtype=np.float64) + y, x
