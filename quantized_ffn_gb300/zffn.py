"""Python binding of libzffn (include/zffn.h): argument marshalling only.

Every function takes CUDA tensors, checks dtype/shape/contiguity, and passes
raw device pointers and the current (or given) CUDA stream to the C ABI.  All
computation happens in the library's kernels; if the library is not built,
importing the functions raises -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libzffn.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_NO_WORKSPACE = range(6)
OPT_MATVEC_MAX_T = 1
OPT_MOE_KERNEL = 2
OPT_TOKEN_KERNEL = 3

_lock = threading.Lock()
_lib = None


class ZffnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        detail = ""
        if status == ERR_CUDA:
            detail = " (" + load().zffn_last_error().decode() + ")"
        super().__init__(f"{what}: {status_string(status)}{detail}")


def load() -> ctypes.CDLL:
    """Load libzffn.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with quantized_ffn_gb300.build.build()")
            lib = ctypes.CDLL(LIB_PATH)
            P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
            sigs = {
                "zffn_status_string": ([I32], ctypes.c_char_p),
                "zffn_last_error": ([], ctypes.c_char_p),
                "zffn_q4k_row_bytes": ([I64], ctypes.c_size_t),
                "zffn_q4k_dequant": ([P, P, I64, I64, P], I32),
                "zffn_q4k_quantize": ([P, P, I64, I64, P], I32),
                "zffn_swiglu_q4k": ([P, P, P, P, P, I32, I32, I32, P], I32),
                "zffn_moe_swiglu_q4k": ([P, P, P, P, P, P, P, I32, I32, I32, I32, I32, P], I32),
                "zffn_swiglu_q4k_residual": ([P, P, P, P, P, I32, I32, I32, P], I32),
                "zffn_moe_swiglu_q4k_residual": ([P, P, P, P, P, P, P, I32, I32, I32, I32, I32, P],
                                                 I32),
                "zffn_moe_router_topk": ([P, P, P, I32, I32, I32, P], I32),
                "zffn_row_bytes_fmt": ([I32, I64], ctypes.c_size_t),
                "zffn_dequant_fmt": ([I32, P, P, I64, I64, P], I32),
                "zffn_swiglu_q4k_wd": ([P, P, P, P, I32, P, I32, I32, I32, P], I32),
                "zffn_moe_swiglu_q4k_wd": ([P, P, P, P, P, P, I32, P, I32, I32, I32, I32, I32, P], I32),
                "zffn_moe_swiglu_q4k_scaled": ([P, P, P, P, P, P, P, I32, P, I32, I32, I32, I32, I32, I32, P],
                                               I32),
                "zffn_rmsnorm_bf16": ([P, P, ctypes.c_float, P, I32, I32, P], I32),
                "zffn_swiglu_q4k_prenorm_residual": ([P, P, ctypes.c_float, P, P, P, I32, I32, I32, P],
                                                     I32),
                "zffn_pipeline_create": ([ctypes.POINTER(ctypes.c_void_p), I32, I32, I32, I32], I32),
                "zffn_pipeline_submit": ([P, P, P, P, P, P], I32),
                "zffn_pipeline_submit_moe": ([P, P, P, P, P, P, P, I32, I32, P], I32),
                "zffn_pipeline_sync": ([P], I32),
                "zffn_pipeline_destroy": ([P], None),
                "zffn_reserve": ([I32, I32, I32, I32, I32], I32),
                "zffn_release": ([], None),
                "zffn_workspace_bytes": ([], ctypes.c_size_t),
                "zffn_single_token_launches": ([I32, I32, I32, I32], I32),
                "zffn_get_device_error": ([P], I32),
                "zffn_set_option": ([I32, I32], I32),
                "zffn_selftest_wait_timeout": ([I64, P], I32),
            }
            for name, (args, res) in sigs.items():
                f = getattr(lib, name)
                f.argtypes = args
                f.restype = res
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().zffn_status_string(int(status)).decode()


def _check(status: int, what: str):
    if status != OK:
        raise ZffnError(status, what)


def _stream(stream: Optional[torch.cuda.Stream]) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _cuda(t: torch.Tensor, name: str, dtype=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def q4k_row_bytes(cols: int) -> int:
    return int(load().zffn_q4k_row_bytes(int(cols)))


def q4k_dequant(blocks: torch.Tensor, rows: int, cols: int, out: Optional[torch.Tensor] = None,
                stream=None) -> torch.Tensor:
    if out is None:
        out = torch.empty((rows, cols), dtype=torch.float32, device=blocks.device)
    if blocks.numel() < rows * q4k_row_bytes(cols):
        raise ValueError("blocks too small")
    _check(load().zffn_q4k_dequant(_cuda(blocks, "blocks", torch.uint8),
                                   _cuda(out, "out", torch.float32), rows, cols, _stream(stream)),
           "zffn_q4k_dequant")
    return out


def q4k_quantize(w: torch.Tensor, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    rows, cols = w.shape
    if out is None:
        out = torch.empty((rows, q4k_row_bytes(cols)), dtype=torch.uint8, device=w.device)
    _check(load().zffn_q4k_quantize(_cuda(w, "w", torch.float32), _cuda(out, "out", torch.uint8),
                                    rows, cols, _stream(stream)), "zffn_q4k_quantize")
    return out


def swiglu_q4k(x: torch.Tensor, Wg: torch.Tensor, Wu: torch.Tensor, Wd: torch.Tensor, I: int,
               y: Optional[torch.Tensor] = None, stream=None, residual: bool = False
               ) -> torch.Tensor:
    """y[T, H] fp32 = W_down (silu(W_gate x) * (W_up x)) with Q4_K weights
    (residual=True: y += that, y must be given)."""
    T, H = x.shape
    if y is None:
        if residual:
            raise ValueError("residual=True needs y")
        y = torch.empty((T, H), dtype=torch.float32, device=x.device)
    fn = load().zffn_swiglu_q4k_residual if residual else load().zffn_swiglu_q4k
    _check(fn(_cuda(x, "x", torch.bfloat16), _cuda(Wg, "Wg", torch.uint8),
              _cuda(Wu, "Wu", torch.uint8), _cuda(Wd, "Wd", torch.uint8),
              _cuda(y, "y", torch.float32), T, H, I, _stream(stream)), "zffn_swiglu_q4k")
    return y


def moe_swiglu_q4k(x: torch.Tensor, expert_ids: torch.Tensor, expert_weights: torch.Tensor,
                   Wg: torch.Tensor, Wu: torch.Tensor, Wd: torch.Tensor, I: int, E: int,
                   y: Optional[torch.Tensor] = None, stream=None, residual: bool = False
                   ) -> torch.Tensor:
    """Routed experts: y[t] = sum_j w[t, j] FFN_{ids[t, j]}(x[t]) (residual: y += ...)."""
    T, H = x.shape
    top_k = expert_ids.shape[1]
    if y is None:
        if residual:
            raise ValueError("residual=True needs y")
        y = torch.empty((T, H), dtype=torch.float32, device=x.device)
    fn = load().zffn_moe_swiglu_q4k_residual if residual else load().zffn_moe_swiglu_q4k
    _check(fn(
        _cuda(x, "x", torch.bfloat16), _cuda(expert_ids, "expert_ids", torch.int32),
        _cuda(expert_weights, "expert_weights", torch.float32), _cuda(Wg, "Wg", torch.uint8),
        _cuda(Wu, "Wu", torch.uint8), _cuda(Wd, "Wd", torch.uint8),
        _cuda(y, "y", torch.float32), T, H, I, E, top_k, _stream(stream)), "zffn_moe_swiglu_q4k")
    return y


FMT_Q4_K, FMT_Q5_K, FMT_Q6_K, FMT_Q5_1 = 0, 1, 2, 3


def row_bytes_fmt(fmt: int, cols: int) -> int:
    return int(load().zffn_row_bytes_fmt(int(fmt), int(cols)))


def dequant_fmt(blocks: torch.Tensor, fmt: int, rows: int, cols: int,
                out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """fp32 [rows, cols] from rows of blocks of format fmt (bit-exact)."""
    if out is None:
        out = torch.empty((rows, cols), dtype=torch.float32, device=blocks.device)
    _check(load().zffn_dequant_fmt(int(fmt), _cuda(blocks, "blocks", torch.uint8),
                                   _cuda(out, "out", torch.float32), rows, cols, _stream(stream)),
           "zffn_dequant_fmt")
    return out


def swiglu_q4k_wd(x: torch.Tensor, Wg: torch.Tensor, Wu: torch.Tensor, Wd: torch.Tensor, wd_fmt: int,
                  I: int, y: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """The block with W_down in block format wd_fmt (zffn_format: Q4_K, Q5_K, Q6_K, Q5_1);
    T = 1 on the single-token kernels, T > 1 on the grouped tensor-core kernel."""
    T, H = x.shape
    if y is None:
        y = torch.empty((T, H), dtype=torch.float32, device=x.device)
    _check(load().zffn_swiglu_q4k_wd(_cuda(x, "x", torch.bfloat16), _cuda(Wg, "Wg", torch.uint8),
                                     _cuda(Wu, "Wu", torch.uint8), _cuda(Wd, "Wd", torch.uint8),
                                     int(wd_fmt), _cuda(y, "y", torch.float32), T, H, I,
                                     _stream(stream)), "zffn_swiglu_q4k_wd")
    return y


def moe_swiglu_q4k_wd(x: torch.Tensor, expert_ids: torch.Tensor, expert_weights: torch.Tensor,
                      Wg: torch.Tensor, Wu: torch.Tensor, Wd: torch.Tensor, wd_fmt: int, I: int,
                      E: int, y: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """The routed block with every expert's W_down in block format wd_fmt."""
    T, H = x.shape
    top_k = expert_ids.shape[1]
    if y is None:
        y = torch.empty((T, H), dtype=torch.float32, device=x.device)
    _check(load().zffn_moe_swiglu_q4k_wd(
        _cuda(x, "x", torch.bfloat16), _cuda(expert_ids, "expert_ids", torch.int32),
        _cuda(expert_weights, "expert_weights", torch.float32), _cuda(Wg, "Wg", torch.uint8),
        _cuda(Wu, "Wu", torch.uint8), _cuda(Wd, "Wd", torch.uint8), int(wd_fmt),
        _cuda(y, "y", torch.float32), T, H, I, E, top_k, _stream(stream)), "zffn_moe_swiglu_q4k_wd")
    return y


def moe_swiglu_q4k_scaled(x: torch.Tensor, expert_ids: torch.Tensor, expert_weights: torch.Tensor,
                          down_scale: Optional[torch.Tensor], Wg: torch.Tensor, Wu: torch.Tensor,
                          Wd: torch.Tensor, I: int, E: int, wd_fmt: int = 0,
                          y: Optional[torch.Tensor] = None, accumulate: bool = False,
                          stream=None) -> torch.Tensor:
    """Routed block with a scale on each expert's down projection:
    y[t] (+)= sum_j w[t, j] * down_scale[ids[t, j]] * FFN_{ids[t, j]}(x[t])
    (down_scale fp32 [E] or None for all ones; W_down in block format wd_fmt)."""
    T, H = x.shape
    top_k = expert_ids.shape[1]
    if y is None:
        if accumulate:
            raise ValueError("accumulate=True needs y")
        y = torch.empty((T, H), dtype=torch.float32, device=x.device)
    sc = None
    if down_scale is not None:
        if down_scale.numel() != E:
            raise ValueError("down_scale must hold E values")
        sc = _cuda(down_scale, "down_scale", torch.float32)
    _check(load().zffn_moe_swiglu_q4k_scaled(
        _cuda(x, "x", torch.bfloat16), _cuda(expert_ids, "expert_ids", torch.int32),
        _cuda(expert_weights, "expert_weights", torch.float32), sc, _cuda(Wg, "Wg", torch.uint8),
        _cuda(Wu, "Wu", torch.uint8), _cuda(Wd, "Wd", torch.uint8), int(wd_fmt),
        _cuda(y, "y", torch.float32), T, H, I, E, top_k, int(bool(accumulate)), _stream(stream)),
        "zffn_moe_swiglu_q4k_scaled")
    return y


def rmsnorm_bf16(h: torch.Tensor, gamma: torch.Tensor, eps: float,
                 out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """x[T, H] bf16 = h / sqrt(mean(h^2) + eps) * gamma, row by row (h fp32)."""
    T, H = h.shape
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=h.device)
    _check(load().zffn_rmsnorm_bf16(_cuda(h, "h", torch.float32), _cuda(gamma, "gamma", torch.float32),
                                    float(eps), _cuda(out, "x", torch.bfloat16), T, H, _stream(stream)),
           "zffn_rmsnorm_bf16")
    return out


def swiglu_q4k_prenorm_residual(h: torch.Tensor, gamma: torch.Tensor, eps: float, Wg: torch.Tensor,
                                Wu: torch.Tensor, Wd: torch.Tensor, I: int, stream=None
                                ) -> torch.Tensor:
    """h += W_down (silu(W_gate x) * (W_up x)) with x = rmsnorm_bf16(h, gamma, eps),
    in place on the fp32 residual stream h [T, H]; returns h."""
    T, H = h.shape
    _check(load().zffn_swiglu_q4k_prenorm_residual(
        _cuda(h, "h", torch.float32), _cuda(gamma, "gamma", torch.float32), float(eps),
        _cuda(Wg, "Wg", torch.uint8), _cuda(Wu, "Wu", torch.uint8), _cuda(Wd, "Wd", torch.uint8),
        T, H, I, _stream(stream)), "zffn_swiglu_q4k_prenorm_residual")
    return h


def moe_router_topk(logits: torch.Tensor, top_k: int, expert_ids: Optional[torch.Tensor] = None,
                    expert_weights: Optional[torch.Tensor] = None, stream=None):
    """(expert_ids int32 [T, top_k], expert_weights fp32 [T, top_k]) from
    router logits fp32 [T, E]: the top_k experts of each token (highest logit
    first, ties to the lower index) and softmax weights over the chosen logits."""
    T, E = logits.shape
    if expert_ids is None:
        expert_ids = torch.empty((T, top_k), dtype=torch.int32, device=logits.device)
    if expert_weights is None:
        expert_weights = torch.empty((T, top_k), dtype=torch.float32, device=logits.device)
    _check(load().zffn_moe_router_topk(
        _cuda(logits, "logits", torch.float32), _cuda(expert_ids, "expert_ids", torch.int32),
        _cuda(expert_weights, "expert_weights", torch.float32), T, E, top_k, _stream(stream)),
        "zffn_moe_router_topk")
    return expert_ids, expert_weights


def _host(t: torch.Tensor, name: str, dtype, shape):
    if t.is_cuda:
        raise ValueError(f"{name} must be a host tensor")
    if t.dtype != dtype or tuple(t.shape) != tuple(shape) or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {dtype} tensor of shape {tuple(shape)}")
    return ctypes.c_void_p(t.data_ptr())


class Pipeline:
    """Dense blocks over host buffers with the copies overlapped (zffn_pipeline_*).

    submit() queues upload(x_host) -> block -> download(y_host) and returns at
    once; sync() waits for everything submitted.  x_host (bf16 [T, H]) and
    y_host (fp32 [T, H]) are CPU tensors, page-locked for the copies to
    overlap, and must stay alive and unchanged until sync() returns."""

    def __init__(self, T: int, H: int, I: int, depth: int = 2):
        self.T, self.H, self.I = T, H, I
        self._p = ctypes.c_void_p()
        _check(load().zffn_pipeline_create(ctypes.byref(self._p), T, H, I, depth),
               "zffn_pipeline_create")
        self._keep = []

    def submit(self, x_host: torch.Tensor, Wg: torch.Tensor, Wu: torch.Tensor, Wd: torch.Tensor,
               y_host: torch.Tensor):
        if not self._p:
            raise RuntimeError("pipeline is closed")
        shape = (self.T, self.H)
        _check(load().zffn_pipeline_submit(
            self._p, _host(x_host, "x_host", torch.bfloat16, shape), _cuda(Wg, "Wg", torch.uint8),
            _cuda(Wu, "Wu", torch.uint8), _cuda(Wd, "Wd", torch.uint8),
            _host(y_host, "y_host", torch.float32, shape)), "zffn_pipeline_submit")
        self._keep.append((x_host, y_host, Wg, Wu, Wd))

    def submit_moe(self, x_host: torch.Tensor, expert_ids: torch.Tensor, expert_weights: torch.Tensor,
                   Wg: torch.Tensor, Wu: torch.Tensor, Wd: torch.Tensor, E: int, y_host: torch.Tensor):
        """The routed block; ids and weights [T, top_k] on the device."""
        if not self._p:
            raise RuntimeError("pipeline is closed")
        shape = (self.T, self.H)
        top_k = expert_ids.shape[1]
        _check(load().zffn_pipeline_submit_moe(
            self._p, _host(x_host, "x_host", torch.bfloat16, shape),
            _cuda(expert_ids, "expert_ids", torch.int32),
            _cuda(expert_weights, "expert_weights", torch.float32), _cuda(Wg, "Wg", torch.uint8),
            _cuda(Wu, "Wu", torch.uint8), _cuda(Wd, "Wd", torch.uint8), E, top_k,
            _host(y_host, "y_host", torch.float32, shape)), "zffn_pipeline_submit_moe")
        self._keep.append((x_host, y_host, expert_ids, expert_weights, Wg, Wu, Wd))

    def sync(self):
        _check(load().zffn_pipeline_sync(self._p), "zffn_pipeline_sync")
        self._keep.clear()

    def close(self):
        if self._p:
            load().zffn_pipeline_destroy(self._p)
            self._p = ctypes.c_void_p()
            self._keep.clear()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def reserve(T_max: int, H_max: int, I_max: int, E_max: int = 1, top_k_max: int = 1):
    _check(load().zffn_reserve(T_max, H_max, I_max, E_max, top_k_max), "zffn_reserve")


def release():
    load().zffn_release()


def workspace_bytes() -> int:
    """Bytes of library workspace held on the current device."""
    return int(load().zffn_workspace_bytes())


def single_token_launches(H: int, I: int, E: int, top_k: int) -> int:
    """Kernel launches of one routed single-token call of these sizes (1: the
    one cooperative launch, 2: the gate/up and down pair; -1 without a device)."""
    return int(load().zffn_single_token_launches(H, I, E, top_k))


def get_device_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error word."""
    return int(load().zffn_get_device_error(_stream(stream)))


def set_option(key: int, value: int) -> int:
    return int(load().zffn_set_option(key, value))


def selftest_wait_timeout(budget_cycles: int, stream=None):
    _check(load().zffn_selftest_wait_timeout(int(budget_cycles), _stream(stream)),
           "zffn_selftest_wait_timeout")
