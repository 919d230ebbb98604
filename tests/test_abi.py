"""The C ABI on the host (no GPU): the library loads, exports every function
declared in include/zffn.h, and rejects invalid arguments before touching the
device."""
import ctypes
import os
import re

import pytest
import torch

from quantized_ffn_gb300 import build as zbuild
from quantized_ffn_gb300 import zffn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    zbuild.build()
    return zffn.load()


def declared_functions():
    names = []
    with open(os.path.join(ROOT, "include", "zffn.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    for m in re.finditer(r"\b(zffn_\w+)\s*\(", text):
        names.append(m.group(1))
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("zffn_q4k_dequant", "zffn_swiglu_q4k", "zffn_moe_swiglu_q4k"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code, name in enumerate(["ZFFN_OK", "ZFFN_ERR_INVALID_ARG", "ZFFN_ERR_UNSUPPORTED",
                                 "ZFFN_ERR_CUDA", "ZFFN_ERR_TIMEOUT", "ZFFN_ERR_NO_WORKSPACE"]):
        assert zffn.status_string(code) == name


def test_row_bytes(lib):
    assert zffn.q4k_row_bytes(256) == 144
    assert zffn.q4k_row_bytes(4096) == 16 * 144
    assert zffn.q4k_row_bytes(11008) == 43 * 144
    assert zffn.q4k_row_bytes(704) == 3 * 144
    assert zffn.q4k_row_bytes(0) == 0


FAKE = ctypes.c_void_p(0x10000)   # never dereferenced: the checks reject first


@pytest.mark.parametrize("T,H,I", [(0, 256, 256), (4, 200, 256), (4, 256, 100), (4, 256, 0),
                                   (4, 32768, 256), (-1, 256, 256)])
def test_swiglu_rejects_bad_shapes(lib, T, H, I):
    st = lib.zffn_swiglu_q4k(FAKE, FAKE, FAKE, FAKE, FAKE, T, H, I, None)
    assert st == zffn.ERR_INVALID_ARG


def test_swiglu_rejects_null_and_misaligned(lib):
    assert lib.zffn_swiglu_q4k(None, FAKE, FAKE, FAKE, FAKE, 4, 256, 256, None) == zffn.ERR_INVALID_ARG
    assert lib.zffn_swiglu_q4k(FAKE, FAKE, FAKE, None, FAKE, 4, 256, 256, None) == zffn.ERR_INVALID_ARG
    odd = ctypes.c_void_p(0x10008)
    assert lib.zffn_swiglu_q4k(odd, FAKE, FAKE, FAKE, FAKE, 4, 256, 256, None) == zffn.ERR_INVALID_ARG


@pytest.mark.parametrize("E,k", [(0, 1), (5000, 1), (8, 0), (8, 65)])
def test_moe_rejects_bad_routing_sizes(lib, E, k):
    st = lib.zffn_moe_swiglu_q4k(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 256, 256, E, k, None)
    assert st == zffn.ERR_INVALID_ARG


def test_dequant_quantize_reject_bad_args(lib):
    assert lib.zffn_q4k_dequant(None, FAKE, 1, 256, None) == zffn.ERR_INVALID_ARG
    assert lib.zffn_q4k_dequant(FAKE, FAKE, 0, 256, None) == zffn.ERR_INVALID_ARG
    assert lib.zffn_q4k_quantize(FAKE, None, 1, 256, None) == zffn.ERR_INVALID_ARG
    assert lib.zffn_q4k_quantize(FAKE, FAKE, 1, -5, None) == zffn.ERR_INVALID_ARG


def test_reserve_and_selftest_reject_bad_args(lib):
    assert lib.zffn_reserve(0, 1, 1, 1, 1) == zffn.ERR_INVALID_ARG
    assert lib.zffn_selftest_wait_timeout(0, None) == zffn.ERR_INVALID_ARG


def test_options(lib):
    old = zffn.set_option(zffn.OPT_MATVEC_MAX_T, 4)
    assert zffn.set_option(zffn.OPT_MATVEC_MAX_T, old) == 4
    assert zffn.set_option(999, 1) == -1
    old = zffn.set_option(zffn.OPT_TOKEN_KERNEL, 1)
    assert zffn.set_option(zffn.OPT_TOKEN_KERNEL, old) == 1


def test_single_token_launch_query_without_device(lib):
    # bad sizes, and (on a host without a GPU) no device: -1
    assert zffn.single_token_launches(2048, 768, 128, 0) == -1
    assert zffn.single_token_launches(2048, 768, 128, 65) == -1
    if not torch.cuda.is_available():
        assert zffn.single_token_launches(2048, 768, 128, 8) == -1


@pytest.mark.parametrize("T,E,k", [(0, 8, 2), (-3, 8, 2), (4, 0, 1), (4, 5000, 8), (4, 8, 0),
                                   (4, 8, 9), (4, 128, 65)])
def test_router_rejects_bad_sizes(lib, T, E, k):
    assert lib.zffn_moe_router_topk(FAKE, FAKE, FAKE, T, E, k, None) == zffn.ERR_INVALID_ARG


def test_router_rejects_null_and_misaligned(lib):
    assert lib.zffn_moe_router_topk(None, FAKE, FAKE, 4, 8, 2, None) == zffn.ERR_INVALID_ARG
    assert lib.zffn_moe_router_topk(FAKE, None, FAKE, 4, 8, 2, None) == zffn.ERR_INVALID_ARG
    assert lib.zffn_moe_router_topk(FAKE, FAKE, None, 4, 8, 2, None) == zffn.ERR_INVALID_ARG
    odd = ctypes.c_void_p(0x10002)
    assert lib.zffn_moe_router_topk(odd, FAKE, FAKE, 4, 8, 2, None) == zffn.ERR_INVALID_ARG


@pytest.mark.parametrize("T,H,eps", [(0, 256, 1e-6), (4, 200, 1e-6), (4, 32768, 1e-6),
                                     (4, 256, -1.0), (4, 256, float("nan")), (4, 256, 2.0)])
def test_rmsnorm_rejects_bad_args(lib, T, H, eps):
    assert lib.zffn_rmsnorm_bf16(FAKE, FAKE, eps, FAKE, T, H, None) == zffn.ERR_INVALID_ARG
    assert lib.zffn_swiglu_q4k_prenorm_residual(FAKE, FAKE, eps, FAKE, FAKE, FAKE, T, H, 256,
                                                None) == zffn.ERR_INVALID_ARG


def test_rmsnorm_rejects_null_and_misaligned(lib):
    odd = ctypes.c_void_p(0x10008)
    assert lib.zffn_rmsnorm_bf16(None, FAKE, 1e-6, FAKE, 4, 256, None) == zffn.ERR_INVALID_ARG
    assert lib.zffn_rmsnorm_bf16(FAKE, odd, 1e-6, FAKE, 4, 256, None) == zffn.ERR_INVALID_ARG
    assert lib.zffn_swiglu_q4k_prenorm_residual(odd, FAKE, 1e-6, FAKE, FAKE, FAKE, 4, 256, 256,
                                                None) == zffn.ERR_INVALID_ARG
    assert lib.zffn_swiglu_q4k_prenorm_residual(FAKE, FAKE, 1e-6, FAKE, None, FAKE, 4, 256, 256,
                                                None) == zffn.ERR_INVALID_ARG


@pytest.mark.parametrize("T,H,I,depth", [(0, 256, 256, 2), (4, 200, 256, 2), (4, 256, 100, 2),
                                         (4, 256, 256, 1), (4, 256, 256, 5)])
def test_pipeline_rejects_bad_args(lib, T, H, I, depth):
    p = ctypes.c_void_p(1)
    assert zffn.load().zffn_pipeline_create(ctypes.byref(p), T, H, I, depth) == zffn.ERR_INVALID_ARG
    assert not p.value
    assert zffn.load().zffn_pipeline_create(None, 4, 256, 256, 2) == zffn.ERR_INVALID_ARG
    assert zffn.load().zffn_pipeline_submit(None, FAKE, FAKE, FAKE, FAKE, FAKE) == zffn.ERR_INVALID_ARG
    assert zffn.load().zffn_pipeline_sync(None) == zffn.ERR_INVALID_ARG
    zffn.load().zffn_pipeline_destroy(None)


def test_format_row_bytes_and_rejections(lib):
    assert zffn.row_bytes_fmt(zffn.FMT_Q4_K, 11008) == 43 * 144
    assert zffn.row_bytes_fmt(zffn.FMT_Q5_K, 768) == 3 * 176
    assert zffn.row_bytes_fmt(zffn.FMT_Q6_K, 11008) == 43 * 210
    assert zffn.row_bytes_fmt(zffn.FMT_Q5_1, 704) == 22 * 24
    assert zffn.row_bytes_fmt(7, 256) == 0 and zffn.row_bytes_fmt(zffn.FMT_Q5_K, 0) == 0
    L = lib
    assert L.zffn_dequant_fmt(7, FAKE, FAKE, 1, 256, None) == zffn.ERR_INVALID_ARG
    assert L.zffn_dequant_fmt(1, FAKE, FAKE, 0, 256, None) == zffn.ERR_INVALID_ARG
    assert L.zffn_swiglu_q4k_wd(FAKE, FAKE, FAKE, FAKE, 9, FAKE, 1, 256, 256, None) == zffn.ERR_INVALID_ARG
    assert L.zffn_swiglu_q4k_wd(FAKE, FAKE, FAKE, FAKE, 2, FAKE, 1, 200, 256, None) == zffn.ERR_INVALID_ARG
    # every format at T > 1 wants a 16-byte aligned W_down (checked on the host)
    odd4 = ctypes.c_void_p(0x10004)
    for fmt in (1, 2, 3):
        assert L.zffn_swiglu_q4k_wd(FAKE, FAKE, FAKE, odd4, fmt, FAKE, 4, 256, 256, None) == zffn.ERR_INVALID_ARG
        assert L.zffn_moe_swiglu_q4k_wd(FAKE, FAKE, FAKE, FAKE, FAKE, odd4, fmt, FAKE, 3, 256, 256, 8, 2,
                                        None) == zffn.ERR_INVALID_ARG
    assert L.zffn_moe_swiglu_q4k_wd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, FAKE, 1, 256, 256, 0, 2,
                                    None) == zffn.ERR_INVALID_ARG


def declared_signatures():
    """{name: (return type, parameter count)} from include/zffn.h."""
    with open(os.path.join(ROOT, "include", "zffn.h")) as f:
        text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
    sigs = {}
    for m in re.finditer(r"([A-Za-z_][\w\s\*]*?)\b(zffn_\w+)\s*\(([^)]*)\)\s*;", text):
        ret, name, params = m.group(1).strip(), m.group(2), m.group(3).strip()
        n = 0 if params in ("", "void") else len(params.split(","))
        sigs[name] = (ret, n)
    return sigs


def test_binding_signatures_match_the_header(lib):
    # every function the binding types must have the header's arity and
    # return type class
    sigs = declared_signatures()
    assert "zffn_swiglu_q4k" in sigs and sigs["zffn_swiglu_q4k"][1] == 9
    checked = 0
    for name, (ret, n) in sigs.items():
        f = getattr(lib, name)
        if f.argtypes is None:
            continue                     # called through ctypes directly by its test
        checked += 1
        assert len(f.argtypes) == n, (name, len(f.argtypes), n)
        if ret.startswith("zffn_status") or ret == "int":
            assert f.restype is ctypes.c_int, name
        elif ret.startswith("size_t"):
            assert f.restype is ctypes.c_size_t, name
        elif ret.startswith("void"):
            assert f.restype is None, name
        elif "char" in ret:
            assert f.restype is ctypes.c_char_p, name
    assert checked >= 25


def test_header_compiles_as_plain_c(tmp_path):
    # the boundary is a C ABI: the header must compile as C99 without warnings
    src = tmp_path / "use.c"
    src.write_text(
        '#include "zffn.h"\n'
        "int use(const void *x, const void *w, float *y, void *s) {\n"
        "    zffn_pipeline *p = 0;\n"
        "    size_t rb = zffn_q4k_row_bytes(4096) + zffn_row_bytes_fmt(ZFFN_FMT_Q6_K, 11008);\n"
        "    zffn_status st = zffn_swiglu_q4k(x, w, w, w, y, 1, 4096, 11008, s);\n"
        "    if (zffn_pipeline_create(&p, 1, 4096, 11008, 2) == ZFFN_OK) zffn_pipeline_destroy(p);\n"
        "    return (int)st + (int)rb + (zffn_status_string(st) != 0);\n"
        "}\n")
    import subprocess
    subprocess.check_call(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                           "-I", os.path.join(ROOT, "include"), "-c", str(src), "-o",
                           str(tmp_path / "use.o")])


def test_rejections_record_the_failed_check(lib):
    st = lib.zffn_swiglu_q4k(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 200, 256, None)
    assert st == zffn.ERR_INVALID_ARG and b"H must be" in lib.zffn_last_error()
    odd = ctypes.c_void_p(0x10008)
    st = lib.zffn_swiglu_q4k(odd, FAKE, FAKE, FAKE, FAKE, 4, 256, 256, None)
    assert st == zffn.ERR_INVALID_ARG and b"aligned" in lib.zffn_last_error()
    st = lib.zffn_moe_swiglu_q4k(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 256, 256, 8, 0, None)
    assert st == zffn.ERR_INVALID_ARG and b"top_k" in lib.zffn_last_error()


def test_workspace_query_is_zero_before_any_call(lib):
    # in a fresh process, so that no earlier call of this one counts
    import subprocess
    import sys
    code = "from quantized_ffn_gb300 import zffn; print(zffn.workspace_bytes())"
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.split()[-1] == "0", r.stdout


def test_no_device_failure_records_its_reason(lib):
    # well-formed arguments on a host without a GPU: the device lookup fails,
    # the call returns ZFFN_ERR_CUDA and zffn_last_error gives the runtime's text
    if torch.cuda.is_available() or zffn.single_token_launches(2048, 768, 128, 8) != -1:
        pytest.skip("a device is present: the call would launch on the fake pointers")
    lib.zffn_swiglu_q4k(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 200, 256, None)
    assert b"H must be" in lib.zffn_last_error()
    assert lib.zffn_q4k_dequant(FAKE, FAKE, 1, 256, None) == zffn.ERR_CUDA
    msg = lib.zffn_last_error()
    assert msg and msg != b"no error" and b"H must be" not in msg
    assert lib.zffn_swiglu_q4k_token_static(FAKE, FAKE, FAKE, FAKE, FAKE, 256, 256, None) == zffn.ERR_CUDA
    assert lib.zffn_last_error() == msg


def test_routed_entry_rejects_its_own_limits(lib):
    # T * top_k above 2^24, and expert ids or weights not 4-byte aligned
    st = lib.zffn_moe_swiglu_q4k(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, (1 << 18) + 1, 256, 256,
                                 128, 64, None)
    assert st == zffn.ERR_INVALID_ARG and b"2^24" in lib.zffn_last_error()
    odd = ctypes.c_void_p(0x10002)
    for ids, wts in ((odd, FAKE), (FAKE, odd)):
        st = lib.zffn_moe_swiglu_q4k(FAKE, ids, wts, FAKE, FAKE, FAKE, FAKE, 4, 256, 256, 8, 2, None)
        assert st == zffn.ERR_INVALID_ARG and b"4-byte" in lib.zffn_last_error()
