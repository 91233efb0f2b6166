"""The C ABI library loads and exports what include/gdn.h declares; host-side argument
checks answer without touching a GPU (CPU only: no compute calls)."""
import ctypes
import os
import re

import pytest

from gated_deltanet_linear_rule_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "gdn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z_]+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(binding.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_version_and_status_strings(lib):
    assert binding.version() == 10000
    assert binding.status_string(0) == "ok"
    assert binding.status_string(-2) == "pool full"
    for code, text in binding.STATUS.items():
        assert binding.status_string(code) == text


def _shape(**kw):
    base = dict(hqk=16, hv=32, dk=128, dv=128, conv_w=4, chunk=64, io_dtype=1, out_dtype=1, l2_eps=1e-6,
                norm_eps=1e-6, max_prefill_tokens=0)
    base.update(kw)
    return binding.GdnShape(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(hqk=0), -1), (dict(hv=24, hqk=16), -1), (dict(conv_w=0), -1), (dict(conv_w=9), -1),
    (dict(io_dtype=2), -1), (dict(l2_eps=-1.0), -1), (dict(chunk=-1), -1),
    (dict(dk=96, dv=96), -6), (dict(dk=128, dv=64), -6), (dict(chunk=48), -6),
])
def test_pool_create_rejects_bad_shapes_before_any_gpu_work(lib, kw, code):
    h = ctypes.c_void_p()
    assert lib.gdn_pool_create(ctypes.byref(_shape(**kw)), 4, 1, ctypes.byref(h)) == code
    assert not h.value


def test_null_arguments_are_rejected(lib):
    h = ctypes.c_void_p()
    assert lib.gdn_pool_create(None, 4, 1, ctypes.byref(h)) == -1
    assert lib.gdn_pool_create(ctypes.byref(_shape()), 0, 1, ctypes.byref(h)) == -1
    assert lib.gdn_pool_create(ctypes.byref(_shape()), 4, 0, ctypes.byref(h)) == -1
    assert lib.gdn_pool_destroy(None) == -1
    assert lib.gdn_pool_reset(None, None) == -1
    sid = ctypes.c_int()
    assert lib.gdn_slot_alloc(None, ctypes.byref(sid)) == -1
    assert lib.gdn_slot_recycle(None, 0, None) == -1
    assert lib.gdn_slot_ptrs(None, 0, None, 1, None, None) == -1
    assert lib.gdn_layer_params(None, 0, None, None, None, None) == -1
    assert lib.gdn_decode_step(None, 0, None, 1, *([None] * 8)) == -1
    assert lib.gdn_prefill_varlen(None, 0, None, None, 1, 1, *([None] * 8)) == -1
    assert lib.gdn_mixed_step(None, 0, None, 1, *([None] * 7), None, None, 1, 1, *([None] * 7), None) == -1
    assert lib.gdn_last_device_status(None, None) == -1
    assert lib.gdn_pool_get_info(None, None) == -1


def test_noalloc_prefill_rejects_misaligned_rows_before_any_gpu_work(lib):
    """Row buffers are moved in 16-B pieces (and by tensor copies at d = 128): a base address that is not
    16-B aligned is refused by the host checks.  The pointers here are never dereferenced."""
    f = lib.gdn_prefill_varlen_noalloc
    f.restype = ctypes.c_int
    P = ctypes.c_void_p
    good, bad = P(0x100000), P(0x100008)
    args = lambda q: (ctypes.byref(_shape()), good, good, good, good, good, 4, good, good, 1, 64,
                      q, good, good, good, good, good, good, None, None)
    assert f(*args(bad)) == -1
