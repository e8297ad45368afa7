"""The C-ABI library builds, loads and exports every entry point its header declares.

These run without a GPU: only host-side logic is called (version, status names,
workspace sizing, argument validation that rejects a call before any CUDA work).
"""
import ctypes
import os
import re

import pytest

from paged_gqa_attention_gb300 import build as pa_build
from paged_gqa_attention_gb300 import ops

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pagedattn.h")


@pytest.fixture(scope="module")
def lib():
    pa_build.build()
    return ops.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([A-Za-z_][A-Za-z0-9_]*)\s*\(",
                       text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while")))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("kv_append", "paged_attn_decode", "paged_attn_prefill", "pa_workspace_bytes",
                 "pa_check_error", "pa_workspace_init"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"libpagedattn.so does not export {name}"


def test_exports_are_plain_c_symbols(lib):
    out = os.popen(f"nm -D --defined-only {ops.library_path()}").read()
    for name in declared_functions():
        assert re.search(rf"\bT {name}$", out, flags=re.M), f"{name} is not an unmangled text symbol"


def test_version_and_status_strings(lib):
    assert lib.pa_version() == 10000
    for code, name in ops.STATUS.items():
        assert lib.pa_status_string(code).decode() == name


def test_workspace_sizing(lib):
    shape = ops.SHAPE
    n1 = lib.pa_workspace_bytes(shape, 1, 2)
    n32 = lib.pa_workspace_bytes(shape, 32, 16)
    n128 = lib.pa_workspace_bytes(shape, 128, 128)
    assert 0 < n1 <= n32 <= n128
    # header + counters + at most (4096 + 8 * batch) partial entries of 2080 bytes
    assert n128 <= 256 + 4 * 8192 * 8 + (4096 + 8 * 128) * 2080
    bad = ops.pa_shape(32, 4, 128, 256)
    assert lib.pa_workspace_bytes(bad, 1, 1) == 0
    assert lib.pa_workspace_bytes(shape, 0, 1) == 0


def test_host_validation_rejects_before_any_cuda_work(lib):
    null = None
    bad_shape = ops.pa_shape(32, 8, 64, 256)
    # unsupported shape
    assert lib.kv_append(bad_shape, null, null, null, null, null, 1, 1, null, null, 0, 0, null, 0,
                         null) == 2
    assert lib.paged_attn_decode(bad_shape, null, null, null, null, null, null, 1, 1, null, 1,
                                 0.1, null, 0, null) == 2
    assert lib.paged_attn_prefill(bad_shape, null, null, null, null, null, null, 1, 1, null, null,
                                  1, 1, 1, 0.1, null, 0, null) == 2
    # missing workspace
    assert lib.kv_append(ops.SHAPE, null, null, null, null, null, 1, 1, null, null, 1, 1, null, 0,
                         null) == 1
    # negative sizes
    assert lib.paged_attn_decode(ops.SHAPE, null, null, null, null, null, null, 1, 1, null, -1,
                                 0.1, null, 0, null) == 1
    # split length not a multiple of 64
    assert lib.paged_attn_decode_split(ops.SHAPE, null, null, null, null, null, null, 1, 1, null,
                                       1, 0.1, 100, null, 0, null) == 1
    # max_q_len larger than the token count
    assert lib.paged_attn_prefill(ops.SHAPE, null, null, null, null, null, null, 1, 1, null, null,
                                  1, 4, 8, 0.1, null, 0, null) == 1


def test_empty_calls_are_no_ops(lib):
    ws = (ctypes.c_uint8 * 4096)()
    wsp = ctypes.cast(ws, ctypes.c_void_p)
    addr = ctypes.addressof(ws)
    if addr % 16:
        pytest.skip("host buffer not 16-byte aligned")
    # nothing to do -> PA_OK without touching the device
    assert lib.kv_append(ops.SHAPE, None, None, None, None, None, 1, 1, None, None, 0, 0, wsp, 4096,
                         None) == 0
    assert lib.paged_attn_prefill(ops.SHAPE, None, None, None, None, None, None, 1, 1, None, None,
                                  0, 0, 0, 0.1, wsp, 4096, None) == 0


def test_prefill_output_must_be_32_byte_aligned(lib):
    """The prefill writes whole 32-byte sectors: an out pointer that is 16- but not 32-byte
    aligned is rejected on the host (PA_ERR_INVALID_ARG) before any CUDA work.  (The pointers
    are host addresses, so no call here may get past validation.)"""
    buf = (ctypes.c_uint8 * 8192)()
    base = (ctypes.addressof(buf) + 255) // 256 * 256
    ws = ctypes.c_void_p(base)
    p = lambda off: ctypes.c_void_p(base + 1024 + off)
    args = lambda out: (ops.SHAPE, out, None, p(256), p(512), p(768), p(1024), 1, 1, p(1280), p(1536), 1, 4, 4, 0.1,
                        ws, 1024, None)
    assert lib.paged_attn_prefill(*args(p(16))) == 1
    assert lib.paged_attn_prefill(*args(p(48))) == 1


def test_qknorm_gains_and_eps_are_checked_on_the_host(lib):
    """paged_qkv_append_qknorm rejects a missing or misaligned gain and an eps that is
    negative or not finite (PA_ERR_INVALID_ARG) before any CUDA work.  (Host addresses: no
    call here may get past validation.)"""
    buf = (ctypes.c_uint8 * 8192)()
    base = (ctypes.addressof(buf) + 255) // 256 * 256
    p = lambda off: ctypes.c_void_p(base + 1024 + off)
    args = lambda gq, gk, eps: (ops.SHAPE, 256, 0.0, gq, gk, eps, p(0), p(256), p(512), p(768), p(1024), p(1280),
                                1, 1, p(1536), p(1792), 1, 1, ctypes.c_void_p(base), 1024, None)
    assert lib.paged_qkv_append_qknorm(*args(None, p(2048), 1e-6)) == 1
    assert lib.paged_qkv_append_qknorm(*args(p(2048), None, 1e-6)) == 1
    assert lib.paged_qkv_append_qknorm(*args(p(2056), p(2048), 1e-6)) == 1
    for eps in (-1e-6, float("nan"), float("inf")):
        assert lib.paged_qkv_append_qknorm(*args(p(2048), p(2304), eps)) == 1


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(ops, "_lib", None)
    monkeypatch.setattr(ops, "_LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        ops.load()
