"""The C ABI library: it builds for sm_103a, loads without a GPU, exports
every symbol include/pkv.h declares, and returns its documented codes for
calls that fail host validation (no kernel is launched by any of these)."""
import ctypes
import os
import re
import subprocess

import pytest
import torch

import __graft_entry__
import paged_kv_gqa_qk_gb300 as pkv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pkv.h")


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    return pkv.load_library()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"^\s*PKV_API\s+(?:int|const char\s*\*)\s*(pkv_\w+)\s*\(", text, re.M)


def test_header_declares_the_binding_symbols():
    assert sorted(declared_functions()) == sorted(pkv.ABI_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", pkv.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT\s+(\w+)$", out, re.M))
    for name in declared_functions():
        assert name in exported, name
        assert getattr(lib, name)
    # nothing but the ABI is exported
    assert {s for s in exported if s.startswith("pkv")} == set(declared_functions())


def test_default_config_is_qwen3_8b(lib):
    from test_constants import page_constants
    assert pkv.pkv_config_default().as_dict() == page_constants()


def test_strerror(lib):
    assert pkv.pkv_strerror(0) == "ok"
    assert pkv.pkv_strerror(pkv.PKV_EWORKSPACE) == "workspace too small"
    assert pkv.pkv_strerror(12345) == "unknown error"


def test_null_arguments_are_rejected(lib):
    vp = ctypes.c_void_p
    assert lib.pkv_decode(None, *([None] * 7), 1, 1, None, None, 0, None) == pkv.PKV_EINVAL
    assert lib.pkv_step(None, *([None] * 10), 1, 1, 1, None, None, 0, None) == pkv.PKV_EINVAL
    assert lib.pkv_prefill(None, *([None] * 9), 1, 1, 1, None, None, 0, None) == pkv.PKV_EINVAL
    assert lib.pkv_linear(None, None, None, None, 1, 64, 128, None, 0, None) == pkv.PKV_EINVAL
    n = ctypes.c_size_t()
    assert lib.pkv_linear_workspace_bytes(None, 1, 64, 128, ctypes.byref(n)) == pkv.PKV_EINVAL
    assert lib.pkv_workspace_bytes(None, 1, 1, 0, ctypes.byref(n)) == pkv.PKV_EINVAL
    assert lib.pkv_pool_free(None) == pkv.PKV_OK
    assert lib.pkv_pool_kv(None, None, None, None) == pkv.PKV_EINVAL
    assert lib.pkv_check_errors(None, None, None) == pkv.PKV_EINVAL
    assert lib.pkv_set_ctas(None, 0) == pkv.PKV_EINVAL
    assert lib.pkv_timer_enable(None, 1) == pkv.PKV_EINVAL
    assert lib.pkv_config_default(None) == pkv.PKV_EINVAL
    out = vp()
    assert lib.pkv_pool_alloc(None, 8, None, ctypes.byref(out)) == pkv.PKV_EINVAL
    cfg = pkv.pkv_config_default()
    assert lib.pkv_pool_alloc(ctypes.byref(cfg), 0, None, ctypes.byref(out)) == pkv.PKV_EINVAL
    assert lib.pkv_pool_wrap(ctypes.byref(cfg), 8, None, None, None, ctypes.byref(out)) == pkv.PKV_EINVAL
    # misaligned borrowed K/V
    assert lib.pkv_pool_wrap(ctypes.byref(cfg), 8, vp(0x1008), vp(0x2000), None, ctypes.byref(out)) == pkv.PKV_EINVAL


def test_bad_configs_are_rejected(lib):
    out = ctypes.c_void_p()
    for change, code in [(dict(heads=30), pkv.PKV_EINVAL), (dict(head_dim=127), pkv.PKV_EINVAL),
                         (dict(rope_theta=-1.0), pkv.PKV_EINVAL), (dict(eps=float("nan")), pkv.PKV_EINVAL),
                         (dict(head_dim=64), pkv.PKV_ENOTIMPL), (dict(page_size=32), pkv.PKV_ENOTIMPL),
                         (dict(heads=64), pkv.PKV_ENOTIMPL), (dict(max_seq=1 << 21), pkv.PKV_ERANGE)]:
        cfg = pkv.pkv_config_default()
        for k, v in change.items():
            setattr(cfg, k, v)
        assert lib.pkv_pool_alloc(ctypes.byref(cfg), 8, None, ctypes.byref(out)) == code, change
    cfg = pkv.pkv_config_default()
    assert lib.pkv_pool_alloc(ctypes.byref(cfg), 1 << 26, None, ctypes.byref(out)) == pkv.PKV_ERANGE


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_no_device_is_reported(lib):
    out = ctypes.c_void_p()
    cfg = pkv.pkv_config_default()
    assert lib.pkv_pool_alloc(ctypes.byref(cfg), 8, None, ctypes.byref(out)) == pkv.PKV_EDEVICE


def test_missing_library_fails_loudly():
    """No CPU fallback: without libpkv.so the binding raises instead of computing anything."""
    p = subprocess.run(
        [__import__("sys").executable, "-c",
         "import paged_kv_gqa_qk_gb300 as pkv\n"
         "try:\n"
         "    pkv.load_library('/nonexistent/libpkv.so')\n"
         "except RuntimeError as e:\n"
         "    print('raised', e)\n"],
        cwd=ROOT, capture_output=True, text=True, timeout=120)
    assert p.returncode == 0 and p.stdout.startswith("raised") and "libpkv.so not found" in p.stdout
