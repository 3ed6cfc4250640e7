"""ctypes binding of libmla's C ABI (include/mla.h).

The Python names match the C names. Arguments are marshalled only: tensors
become device pointers and streams become cudaStream_t handles. Every step
of the decode path runs in libmla's CUDA kernels. When the library is
missing, :func:`load` raises. There is no Python or CPU fallback.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

MLA_OK = 0
STATUS_NAMES = ["MLA_OK", "MLA_ERR_INVALID_ARG", "MLA_ERR_SHAPE", "MLA_ERR_CAPACITY",
                "MLA_ERR_UNSUPPORTED", "MLA_ERR_WORKSPACE", "MLA_ERR_CUDA",
                "MLA_ERR_DEVICE_CHECK", "MLA_ERR_TIMEOUT"]
MLA_F32, MLA_BF16 = 0, 1
MLA_IMPL_AUTO, MLA_IMPL_CUDA_CORE, MLA_IMPL_TENSOR_CORE = 0, 1, 2
MLA_DEVERR_PAGE_RANGE, MLA_DEVERR_SEQ_LEN, MLA_DEVERR_APPEND_INDEX, MLA_DEVERR_TIMEOUT = 1, 2, 4, 8

# Every symbol include/mla.h declares (checked by the CPU tests).
EXPORTS = ["mla_absorb_weights", "mla_weights_free", "mla_append_kv",
           "mla_decode_workspace_size", "mla_decode", "mla_decode_absorb_q",
           "mla_decode_attend", "mla_decode_combine", "mla_decode_impl",
           "mla_get_last_device_error", "mla_status_string", "mla_decode_no_alloc",
           "mla_fold_full", "mla_full_weights_free", "mla_decode_full_workspace_size",
           "mla_decode_full", "mla_decode_layer_workspace_size", "mla_decode_layer",
           "mla_quantize_rows_fp8", "mla_append_kv_fp8_workspace_size", "mla_append_kv_fp8",
           "mla_decode_fp8", "mla_decode_latent"]
MLA_NO_ALLOC_WORKSPACE_BYTES = 32 << 20


class mla_config(ctypes.Structure):
    _fields_ = [("n_h", ctypes.c_int32), ("d_model", ctypes.c_int32), ("d_c", ctypes.c_int32),
                ("d_r", ctypes.c_int32), ("d_nope", ctypes.c_int32), ("d_v", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("rope_base", ctypes.c_float),
                ("softmax_scale", ctypes.c_float), ("dtype", ctypes.c_int32),
                ("impl", ctypes.c_int32)]


class MlaError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        name = STATUS_NAMES[status] if 0 <= status < len(STATUS_NAMES) else str(status)
        super().__init__(f"{fn} returned {name}")


_P = ctypes.c_void_p
_I = ctypes.c_int32
_lib = None


def _declare(lib):
    cfgp = ctypes.POINTER(mla_config)
    sig = {
        "mla_absorb_weights": [cfgp, _P, _P, _P, _P, _P, ctypes.POINTER(_P)],
        "mla_weights_free": [_P],
        "mla_append_kv": [cfgp, _P, _P, _P, _P, _P, _I, _I, _P, _I, _I, _P],
        "mla_decode_workspace_size": [cfgp, _I, _I, ctypes.c_int64, ctypes.POINTER(ctypes.c_size_t)],
        "mla_decode": [cfgp, _P, _P, _P, _I, _P, _I, _P, _I, _I, _P, _P, ctypes.c_size_t, _P],
        "mla_decode_absorb_q": [cfgp, _P, _P, _P, _I, _I, _I, _P, ctypes.c_size_t, _P],
        "mla_decode_attend": [cfgp, _P, _I, _P, _I, _P, _I, _I, _P, ctypes.c_size_t, _P],
        "mla_decode_latent": [cfgp, _P, _P, _I, _P, _I, _P, _I, _I, _P, _P, ctypes.c_size_t, _P],
        "mla_decode_combine": [cfgp, _P, _P, _I, _I, _P, _P, ctypes.c_size_t, _P],
        "mla_decode_impl": [cfgp, ctypes.POINTER(_I)],
        "mla_decode_no_alloc": [cfgp, _P, _P, _P, _I, _P, _I, _P, _I, _I, _P, _P],
        "mla_fold_full": [cfgp, _P, _P, _P, _P, _P, ctypes.POINTER(_P)],
        "mla_full_weights_free": [_P],
        "mla_decode_full_workspace_size": [cfgp, _I, _I, ctypes.POINTER(ctypes.c_size_t)],
        "mla_decode_full": [cfgp, _P, _P, _P, _I, _P, _I, _P, _I, _I, _P, _P, ctypes.c_size_t, _P],
        "mla_decode_layer_workspace_size": [cfgp, _I, _I, ctypes.POINTER(ctypes.c_size_t)],
        "mla_decode_layer": [cfgp, _P, _P, _P, _P, _P, _P, _P, _I, _P, _I, _P, _I, _I, _P, _P, _P,
                             ctypes.c_size_t, _P],
        "mla_quantize_rows_fp8": [cfgp, _P, _P, _P, _P, _I, _I, _P, _P, _I, _I, _P],
        "mla_append_kv_fp8_workspace_size": [cfgp, _I, ctypes.POINTER(ctypes.c_size_t)],
        "mla_append_kv_fp8": [cfgp, _P, _P, _P, _P, _P, _I, _I, _P, _P, _I, _I, _P,
                              ctypes.c_size_t, _P],
        "mla_decode_fp8": [cfgp, _P, _P, _P, _P, _I, _P, _I, _P, _I, _I, _P, _P, ctypes.c_size_t,
                           _P],
        "mla_get_last_device_error": [_P, ctypes.POINTER(ctypes.c_uint32)],
        "mla_status_string": [_I],
    }
    for name, args in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = ctypes.c_char_p if name == "mla_status_string" else ctypes.c_int


def load(build_if_missing=False):
    """Load libmla.so (built in-tree next to this file)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_build.LIB) or (build_if_missing and not _build.up_to_date()):
        if not build_if_missing:
            raise RuntimeError(f"libmla.so is not built ({_build.LIB}); run "
                               "python -m mla_latent_kv_73_b300.build")
        _build.build()
    lib = ctypes.CDLL(_build.LIB)
    _declare(lib)
    _lib = lib
    return lib


def path():
    return _build.LIB


def check(fn, status):
    if status != MLA_OK:
        raise MlaError(fn, status)


def ptr(t):
    """Device (or host) address of a tensor, or None."""
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def stream_handle(stream):
    """cudaStream_t of a torch.cuda.Stream (None -> the current stream)."""
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def make_config(n_h, d_model, d_c, d_r, d_nope, d_v, block_size=64, rope_base=10000.0,
                softmax_scale=0.0, dtype="bf16", impl=MLA_IMPL_AUTO):
    return mla_config(n_h, d_model, d_c, d_r, d_nope, d_v, block_size, rope_base, softmax_scale,
                      MLA_F32 if dtype in ("f32", "fp32", "float32") else MLA_BF16, impl)


# ------------------------------------------------------------------ wrappers
def mla_absorb_weights(cfg, W_dkv, W_kr, W_uk, W_uv, stream=None):
    lib = load()
    h = ctypes.c_void_p()
    check("mla_absorb_weights", lib.mla_absorb_weights(
        ctypes.byref(cfg), ptr(W_dkv), ptr(W_kr), ptr(W_uk), ptr(W_uv), stream_handle(stream),
        ctypes.byref(h)))
    return h


def mla_weights_free(h):
    check("mla_weights_free", load().mla_weights_free(h))


def mla_append_kv(cfg, w, x, seq_idx, pos, page_table, cache, stream=None):
    B, max_blocks = page_table.shape
    num_blocks = cache.shape[0]
    T = x.shape[0]
    check("mla_append_kv", load().mla_append_kv(
        ctypes.byref(cfg), w, ptr(x), ptr(seq_idx), ptr(pos), ptr(page_table), B, max_blocks,
        ptr(cache), num_blocks, T, stream_handle(stream)))


def mla_decode_workspace_size(cfg, B, n_q, total_tokens=0):
    n = ctypes.c_size_t()
    check("mla_decode_workspace_size", load().mla_decode_workspace_size(
        ctypes.byref(cfg), B, n_q, total_tokens, ctypes.byref(n)))
    return n.value


def mla_decode(cfg, w, q, cache, page_table, seq_lens, out, workspace, stream=None):
    B, n_q = q.shape[0], q.shape[1]
    check("mla_decode", load().mla_decode(
        ctypes.byref(cfg), w, ptr(q), ptr(cache), cache.shape[0], ptr(page_table),
        page_table.shape[1], ptr(seq_lens), B, n_q, ptr(out), ptr(workspace),
        workspace.numel() * workspace.element_size(), stream_handle(stream)))


def mla_quantize_rows_fp8(cfg, rows, seq_idx, pos, page_table, cache, row_scale, stream=None):
    """fp32 rows [T, R] -> e4m3 codes and row scales in the paged fp8 cache."""
    B, max_blocks = page_table.shape
    check("mla_quantize_rows_fp8", load().mla_quantize_rows_fp8(
        ctypes.byref(cfg), ptr(rows), ptr(seq_idx), ptr(pos), ptr(page_table), B, max_blocks,
        ptr(cache), ptr(row_scale), cache.shape[0], rows.shape[0], stream_handle(stream)))


def mla_append_kv_fp8_workspace_size(cfg, T):
    n = ctypes.c_size_t()
    check("mla_append_kv_fp8_workspace_size", load().mla_append_kv_fp8_workspace_size(
        ctypes.byref(cfg), T, ctypes.byref(n)))
    return n.value


def mla_append_kv_fp8(cfg, w, x, seq_idx, pos, page_table, cache, row_scale, workspace,
                      stream=None):
    B, max_blocks = page_table.shape
    check("mla_append_kv_fp8", load().mla_append_kv_fp8(
        ctypes.byref(cfg), w, ptr(x), ptr(seq_idx), ptr(pos), ptr(page_table), B, max_blocks,
        ptr(cache), ptr(row_scale), cache.shape[0], x.shape[0], ptr(workspace),
        workspace.numel() * workspace.element_size(), stream_handle(stream)))


def mla_decode_fp8(cfg, w, q, cache, row_scale, page_table, seq_lens, out, workspace,
                   stream=None):
    B, n_q = q.shape[0], q.shape[1]
    check("mla_decode_fp8", load().mla_decode_fp8(
        ctypes.byref(cfg), w, ptr(q), ptr(cache), ptr(row_scale), cache.shape[0],
        ptr(page_table), page_table.shape[1], ptr(seq_lens), B, n_q, ptr(out), ptr(workspace),
        workspace.numel() * workspace.element_size(), stream_handle(stream)))


def mla_decode_no_alloc(cfg, w, q, cache, page_table, seq_lens, out, stream=None):
    """mla_decode without a workspace argument (see include/mla.h)."""
    B, n_q = q.shape[0], q.shape[1]
    check("mla_decode_no_alloc", load().mla_decode_no_alloc(
        ctypes.byref(cfg), w, ptr(q), ptr(cache), cache.shape[0], ptr(page_table),
        page_table.shape[1], ptr(seq_lens), B, n_q, ptr(out), stream_handle(stream)))


def mla_decode_absorb_q(cfg, w, q, seq_lens, max_blocks, workspace, stream=None):
    B, n_q = q.shape[0], q.shape[1]
    check("mla_decode_absorb_q", load().mla_decode_absorb_q(
        ctypes.byref(cfg), w, ptr(q), ptr(seq_lens), max_blocks, B, n_q, ptr(workspace),
        workspace.numel() * workspace.element_size(), stream_handle(stream)))


def mla_decode_attend(cfg, cache, page_table, seq_lens, B, n_q, workspace, stream=None):
    check("mla_decode_attend", load().mla_decode_attend(
        ctypes.byref(cfg), ptr(cache), cache.shape[0], ptr(page_table), page_table.shape[1],
        ptr(seq_lens), B, n_q, ptr(workspace), workspace.numel() * workspace.element_size(),
        stream_handle(stream)))


def mla_decode_latent(cfg, q_abs, cache, page_table, seq_lens, o_lat, workspace, stream=None):
    """The attention core alone: q_abs [B, n_q, n_h, d_c + d_r] (absorbed and
    rotated, unscaled) -> o_lat [B, n_q, n_h, d_c] fp32 (see include/mla.h)."""
    B, n_q = q_abs.shape[0], q_abs.shape[1]
    check("mla_decode_latent", load().mla_decode_latent(
        ctypes.byref(cfg), ptr(q_abs), ptr(cache), cache.shape[0], ptr(page_table),
        page_table.shape[1], ptr(seq_lens), B, n_q, ptr(o_lat), ptr(workspace),
        workspace.numel() * workspace.element_size(), stream_handle(stream)))


def mla_decode_combine(cfg, w, seq_lens, B, n_q, out, workspace, stream=None):
    check("mla_decode_combine", load().mla_decode_combine(
        ctypes.byref(cfg), w, ptr(seq_lens), B, n_q, ptr(out), ptr(workspace),
        workspace.numel() * workspace.element_size(), stream_handle(stream)))


def mla_decode_impl(cfg):
    v = _I()
    check("mla_decode_impl", load().mla_decode_impl(ctypes.byref(cfg), ctypes.byref(v)))
    return v.value


def mla_fold_full(cfg, W_q, W_uk, W_uv, W_o, stream=None):
    """Folded weights of the full-fold layer (see include/mla.h)."""
    lib = load()
    h = ctypes.c_void_p()
    check("mla_fold_full", lib.mla_fold_full(
        ctypes.byref(cfg), ptr(W_q), ptr(W_uk), ptr(W_uv), ptr(W_o), stream_handle(stream),
        ctypes.byref(h)))
    return h


def mla_full_weights_free(h):
    check("mla_full_weights_free", load().mla_full_weights_free(h))


def mla_decode_full_workspace_size(cfg, B, n_q):
    n = ctypes.c_size_t()
    check("mla_decode_full_workspace_size", load().mla_decode_full_workspace_size(
        ctypes.byref(cfg), B, n_q, ctypes.byref(n)))
    return n.value


def mla_decode_full(cfg, fw, x_q, cache, page_table, seq_lens, y, workspace, stream=None):
    """y [B, n_q, d_model] from the hidden states x_q [B, n_q, d_model]."""
    B, n_q = x_q.shape[0], x_q.shape[1]
    check("mla_decode_full", load().mla_decode_full(
        ctypes.byref(cfg), fw, ptr(x_q), ptr(cache), cache.shape[0], ptr(page_table),
        page_table.shape[1], ptr(seq_lens), B, n_q, ptr(y), ptr(workspace),
        workspace.numel() * workspace.element_size(), stream_handle(stream)))


def mla_decode_layer_workspace_size(cfg, B, n_q):
    n = ctypes.c_size_t()
    check("mla_decode_layer_workspace_size", load().mla_decode_layer_workspace_size(
        ctypes.byref(cfg), B, n_q, ctypes.byref(n)))
    return n.value


def mla_decode_layer(cfg, w, W_o, x, seq_idx, pos, q, cache, page_table, seq_lens, out, y,
                     workspace, stream=None):
    """Append, decode and output projection of one layer (see include/mla.h)."""
    B, n_q = q.shape[0], q.shape[1]
    check("mla_decode_layer", load().mla_decode_layer(
        ctypes.byref(cfg), w, ptr(W_o), ptr(x), ptr(seq_idx), ptr(pos), ptr(q), ptr(cache),
        cache.shape[0], ptr(page_table), page_table.shape[1], ptr(seq_lens), B, n_q, ptr(out),
        ptr(y), ptr(workspace), workspace.numel() * workspace.element_size(),
        stream_handle(stream)))


def mla_get_last_device_error(stream=None):
    """Returns (status, code) without raising."""
    code = ctypes.c_uint32()
    st = load().mla_get_last_device_error(stream_handle(stream), ctypes.byref(code))
    return st, code.value


def mla_status_string(status):
    return load().mla_status_string(status).decode()
