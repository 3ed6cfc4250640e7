"""The C-ABI library loads and exports what include/mla.h declares (CPU only).

No compute call is made here. The argument checks below all fail before
libmla touches a device, so they run on a machine without a GPU.
"""
import ctypes
import os
import re

import pytest

from mla_latent_kv_73_b300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    with open(os.path.join(ROOT, "include", "mla.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:const\s+char\s*\*|mla_status)\s+(mla_\w+)\s*\(",
                                 text, flags=re.M)))


def test_header_declares_the_bound_functions():
    assert declared_functions() == sorted(_lib.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    # and the symbols are real exported C functions
    raw = ctypes.CDLL(_lib.path())
    for name in declared_functions():
        assert ctypes.cast(getattr(raw, name), ctypes.c_void_p).value


def test_status_strings(lib):
    for i, name in enumerate(_lib.STATUS_NAMES):
        assert _lib.mla_status_string(i) == name
    assert _lib.mla_status_string(99) == "MLA_ERR_UNKNOWN"


def good_cfg(**kw):
    c = _lib.make_config(128, 5120, 512, 64, 128, 128)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


@pytest.mark.parametrize("field,value,status", [
    ("d_r", 3, 2), ("d_r", 0, 2), ("d_c", 513, 2), ("d_c", 1024, 2), ("n_h", 0, 2),
    ("d_v", 1025, 2), ("d_nope", 1025, 2),
    ("block_size", 0, 2), ("dtype", 7, 1), ("impl", 5, 1), ("rope_base", 0.0, 1),
    ("softmax_scale", -1.0, 1),
])
def test_config_checks_before_any_device_work(lib, field, value, status):
    cfg = good_cfg(**{field: value})
    n = ctypes.c_size_t(123)
    st = lib.mla_decode_workspace_size(ctypes.byref(cfg), 4, 1, 0, ctypes.byref(n))
    assert st == status and n.value == 0
    h = ctypes.c_void_p(1)
    st = lib.mla_absorb_weights(ctypes.byref(cfg), None, None, None, None, None, ctypes.byref(h))
    assert st == status and h.value is None


def test_null_and_count_checks(lib):
    cfg = good_cfg()
    n = ctypes.c_size_t()
    assert lib.mla_decode_workspace_size(ctypes.byref(cfg), 0, 1, 0, ctypes.byref(n)) == 2
    assert lib.mla_decode_workspace_size(ctypes.byref(cfg), 4, 0, 0, ctypes.byref(n)) == 2
    assert lib.mla_decode_workspace_size(None, 4, 1, 0, ctypes.byref(n)) == 1
    assert lib.mla_decode_workspace_size(ctypes.byref(cfg), 4, 1, 0, None) == 1
    h = ctypes.c_void_p()
    assert lib.mla_absorb_weights(ctypes.byref(cfg), None, None, None, None, None,
                                  ctypes.byref(h)) == 1
    assert lib.mla_absorb_weights(ctypes.byref(cfg), None, None, None, None, None, None) == 1
    assert lib.mla_append_kv(ctypes.byref(cfg), None, None, None, None, None, 1, 1, None, 1, 1,
                             None) == 1
    assert lib.mla_decode(ctypes.byref(cfg), None, None, None, 1, None, 1, None, 1, 1, None, None,
                          0, None) == 1
    assert lib.mla_weights_free(None) == 0
    assert lib.mla_decode_impl(ctypes.byref(cfg), None) == 1
    # the full-fold calls check their arguments the same way
    assert lib.mla_fold_full(ctypes.byref(cfg), None, None, None, None, None,
                             ctypes.byref(h)) == 1
    assert lib.mla_fold_full(ctypes.byref(cfg), None, None, None, None, None, None) == 1
    bad = good_cfg()
    bad.d_c = 3
    assert lib.mla_fold_full(ctypes.byref(bad), None, None, None, None, None,
                             ctypes.byref(h)) == 2
    assert lib.mla_full_weights_free(None) == 0
    assert lib.mla_decode_full_workspace_size(ctypes.byref(cfg), 0, 1, ctypes.byref(n)) == 2
    assert lib.mla_decode_full_workspace_size(ctypes.byref(cfg), 4, 1, None) == 1
    assert lib.mla_decode_full(ctypes.byref(cfg), None, None, None, 1, None, 1, None, 1, 1, None,
                               None, 0, None) == 1
    assert lib.mla_decode_layer_workspace_size(ctypes.byref(cfg), 4, 0, ctypes.byref(n)) == 2
    assert lib.mla_decode_layer_workspace_size(ctypes.byref(cfg), 4, 1, None) == 1
    assert lib.mla_decode_layer(ctypes.byref(cfg), None, None, None, None, None, None, None, 1,
                                None, 1, None, 1, 1, None, None, None, 0, None) == 1
    assert lib.mla_get_last_device_error(None, None) == 1
    # the attention core alone: null pointers, and an o_lat off its 16-byte
    # alignment (never dereferenced: refused before any device work)
    assert lib.mla_decode_latent(ctypes.byref(cfg), None, None, 1, None, 1, None, 1, 1, None,
                                 None, 0, None) == 1
    fake = ctypes.c_void_p(256)
    assert lib.mla_decode_latent(ctypes.byref(cfg), fake, fake, 1, fake, 1, fake, 1, 1,
                                 ctypes.c_void_p(256 + 4), fake, 1 << 20, None) == 1


def test_no_gpu_means_a_loud_cuda_error(lib):
    """Without a device the library reports MLA_ERR_CUDA; it never falls back."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    cfg = good_cfg()
    n = ctypes.c_size_t()
    assert lib.mla_decode_workspace_size(ctypes.byref(cfg), 4, 1, 0, ctypes.byref(n)) == 6
    v = ctypes.c_int32()
    assert lib.mla_decode_impl(ctypes.byref(cfg), ctypes.byref(v)) == 6
    assert lib.mla_decode_full_workspace_size(ctypes.byref(cfg), 4, 1, ctypes.byref(n)) == 6
