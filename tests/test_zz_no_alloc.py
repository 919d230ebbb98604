"""The allocation-free single-token entry point.

Some callers cannot let a library allocate device memory while it runs (their
own allocator owns the device, or allocation is forbidden after start-up).
zffn_swiglu_q4k_token_static serves them: same kernel as the regular
single-token path, scratch in a fixed array inside the library.  These tests
call it through the C ABI and compare it with the oracle and with the regular
entry point on two calls in a row (the array keeps the previous call's
contents, so the second call checks that nothing stale leaks through), and,
in a fresh process where it is the first call into the library, check that
it leaves the library's workspace unallocated.
"""
import ctypes
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest
import torch

from oracle import oracle as orc
from quantized_ffn_gb300 import build as zbuild
from quantized_ffn_gb300 import synth, zffn
from tests.gpu_util import assert_close

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _static_fn(lib):
    fn = lib.zffn_swiglu_q4k_token_static
    fn.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn


def test_static_scratch_entry_matches_oracle_and_regular_entry_on_two_calls():
    zbuild.build()
    fn = _static_fn(zffn.load())
    H, I = 4096, 11008
    rng = np.random.default_rng(2024)
    Wg_h = synth.random_q4k_blocks(rng, I, H, 1e-2)
    Wu_h = synth.random_q4k_blocks(rng, I, H, 1e-2)
    Wd_h = synth.random_q4k_blocks(rng, H, I, 1e-2)
    dev = lambda a: torch.from_numpy(np.array(a, copy=True)).cuda()  # noqa: E731
    Wg, Wu, Wd = dev(Wg_h), dev(Wu_h), dev(Wd_h)
    stream = torch.cuda.current_stream()
    for call in range(2):
        xb = synth.f32_to_bf16_bits(rng.standard_normal((1, H)).astype(np.float32))
        x = dev(xb.view(np.int16)).view(torch.bfloat16)
        y = torch.full((1, H), float("nan"), dtype=torch.float32, device="cuda")
        st = fn(_ptr(x), _ptr(Wg), _ptr(Wu), _ptr(Wd), _ptr(y), H, I,
                ctypes.c_void_p(stream.cuda_stream))
        assert st == zffn.OK, zffn.status_string(st)
        assert zffn.get_device_error() == zffn.OK
        ref = orc.swiglu_ffn(xb, Wg_h, Wu_h, Wd_h, 1, H, I)
        assert_close(y, ref, f"static entry vs oracle, call {call}")
        y_reg = zffn.swiglu_q4k(x, Wg, Wu, Wd, I)
        assert zffn.get_device_error() == zffn.OK
        assert_close(y, y_reg.cpu().numpy().astype(np.float64), f"static entry vs regular entry, call {call}")


def test_static_scratch_entry_allocates_no_workspace_as_first_call():
    # A fresh process, so that this entry point is the first call into the
    # library: afterwards the library's workspace must still be empty.  Only
    # then does the regular entry run (it allocates), as a cross-check.
    zbuild.build()
    code = textwrap.dedent("""
        import ctypes, sys
        import numpy as np, torch
        sys.path.insert(0, %r)
        from quantized_ffn_gb300 import synth, zffn
        lib = zffn.load()
        fn = lib.zffn_swiglu_q4k_token_static
        fn.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
        fn.restype = ctypes.c_int
        H, I = 1024, 1472
        rng = np.random.default_rng(5)
        dev = lambda a: torch.from_numpy(np.array(a, copy=True)).cuda()
        Wg = dev(synth.random_q4k_blocks(rng, I, H, 1e-2))
        Wu = dev(synth.random_q4k_blocks(rng, I, H, 1e-2))
        Wd = dev(synth.random_q4k_blocks(rng, H, I, 1e-2))
        xb = synth.f32_to_bf16_bits(rng.standard_normal((1, H)).astype(np.float32))
        x = dev(xb.view(np.int16)).view(torch.bfloat16)
        y = torch.zeros((1, H), dtype=torch.float32, device="cuda")
        p = lambda t: ctypes.c_void_p(t.data_ptr())
        st = fn(p(x), p(Wg), p(Wu), p(Wd), p(y), H, I, None)
        assert st == 0, st
        torch.cuda.synchronize()
        assert zffn.get_device_error() == 0
        assert zffn.workspace_bytes() == 0, zffn.workspace_bytes()
        y2 = zffn.swiglu_q4k(x, Wg, Wu, Wd, I)
        torch.cuda.synchronize()
        assert zffn.workspace_bytes() > 0
        assert torch.allclose(y, y2, rtol=1e-5, atol=1e-6)
        print("ok")
    """ % ROOT)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr


def test_static_scratch_entry_rejects_sizes_beyond_its_array():
    lib = zffn.load()
    fn = _static_fn(lib)
    buf = torch.zeros(64, dtype=torch.float32, device="cuda")
    p = _ptr(buf)
    st = fn(p, p, p, p, p, 4096, 16384 + 64, None)
    assert st == zffn.ERR_INVALID_ARG
    assert b"16384" in lib.zffn_last_error()
