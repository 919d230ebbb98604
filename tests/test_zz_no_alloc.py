"""The allocation-free single-token entry point.

Some callers cannot let a library allocate device memory while it runs (their
own allocator owns the device, or allocation is forbidden after start-up).
zffn_swiglu_q4k_token_static serves them: same kernel as the regular
single-token path, scratch in a fixed array inside the library.  This test
calls it through the C ABI and compares it with the regular entry point on two
calls in a row (the array keeps the previous call's contents, so the second
call checks that nothing stale leaks through).
"""
import ctypes

import numpy as np
import pytest
import torch

from quantized_ffn_gb300 import build as zbuild
from quantized_ffn_gb300 import synth, zffn
from tests.gpu_util import assert_close

pytestmark = pytest.mark.gpu


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def test_static_scratch_entry_matches_regular_entry_on_two_calls():
    zbuild.build()
    lib = zffn.load()
    fn = lib.zffn_swiglu_q4k_token_static
    fn.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    H, I = 4096, 11008
    rng = np.random.default_rng(2024)
    dev = lambda a: torch.from_numpy(np.array(a, copy=True)).cuda()  # noqa: E731
    Wg = dev(synth.random_q4k_blocks(rng, I, H, 1e-2))
    Wu = dev(synth.random_q4k_blocks(rng, I, H, 1e-2))
    Wd = dev(synth.random_q4k_blocks(rng, H, I, 1e-2))
    stream = torch.cuda.current_stream()
    for call in range(2):
        xb = synth.f32_to_bf16_bits(rng.standard_normal((1, H)).astype(np.float32))
        x = dev(xb.view(np.int16)).view(torch.bfloat16)
        y_ref = zffn.swiglu_q4k(x, Wg, Wu, Wd, I)
        y = torch.full((1, H), float("nan"), dtype=torch.float32, device="cuda")
        st = fn(_ptr(x), _ptr(Wg), _ptr(Wu), _ptr(Wd), _ptr(y), H, I,
                ctypes.c_void_p(stream.cuda_stream))
        assert st == zffn.OK, zffn.status_string(st)
        assert zffn.get_device_error() == zffn.OK
        assert_close(y, y_ref.cpu().numpy().astype(np.float64), f"static entry, call {call}")


def test_static_scratch_entry_rejects_sizes_beyond_its_array():
    lib = zffn.load()
    fn = lib.zffn_swiglu_q4k_token_static
    fn.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    buf = torch.zeros(64, dtype=torch.float32, device="cuda")
    p = _ptr(buf)
    st = fn(p, p, p, p, p, 4096, 16384 + 64, None)
    assert st == zffn.ERR_INVALID_ARG
    assert b"16384" in lib.zffn_last_error()
