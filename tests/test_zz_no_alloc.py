"""mla_decode_no_alloc: decode without a caller-supplied workspace.

This call is for callers that cannot allocate device memory on the decode
path, such as a serving loop that must never wait on an allocator, or a
runtime that owns all device memory itself. It must give the same result as
mla_decode, call after call, while the library's fixed scratch array keeps
whatever the previous call left in it.

The file sorts last so that a run stopping at the first failure has already
run every other test. It also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest

from mla_latent_kv_73_b300 import _lib, synth
from mla_latent_kv_73_b300.device_inputs import DeviceWeights, config_for, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu(lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    st, code = _lib.mla_get_last_device_error()
    assert code == 0, f"device error word left set: {code:#x}"


def _problem(lens, n_q, n_h=128, dtype="bf16", seed=21, d_c=512, d_r=64, d_nope=128, d_v=128):
    w = synth.Workload(f"noalloc_{seed}", n_h=n_h, d_model=64, d_c=d_c, d_r=d_r, d_nope=d_nope,
                       d_v=d_v, batch=len(lens), n_q=n_q, len_lo=0, len_hi=0, dtype=dtype,
                       seed=seed)
    lens = np.asarray(lens, dtype=np.int32)
    cfg = config_for(w)
    dw = DeviceWeights(w, synth.weights(w), cfg)
    pt, nb = synth.page_table(w, lens)
    store, _ = synth.fill_paged_cache(w, lens, pt, nb)
    _, qs = synth.queries(w)
    return dict(w=w, cfg=cfg, dw=dw, cache=to_device(store, w.dtype), pt=to_device(pt, "i32"),
                sl=to_device(lens, "i32"), q=to_device(qs, w.dtype))


def _close(got, ref, dtype):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(got))
    if dtype == "f32":
        assert np.max(np.abs(got - ref)) <= 1e-4
    else:
        rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
        assert rel <= 5e-3 and np.max(np.abs(got - ref)) <= 2e-2


def test_no_alloc_matches_decode_on_consecutive_calls():
    problems = [_problem((5, 70, 130), 1, seed=21),
                _problem((200, 64), 2, seed=22),
                _problem((2, 65, 130), 2, n_h=4, dtype="f32", seed=23, d_c=32, d_r=8, d_nope=16,
                         d_v=16)]
    first = None
    # the first problem runs again last, after larger plans (more splits,
    # more queries) have left their partials in the shared array
    for k, p in enumerate(problems + problems[:1]):
        w = p["w"]
        shape = (w.batch, w.n_q, w.n_h, w.d_v)
        ref = torch.full(shape, float("nan"), device="cuda")
        ws = torch.empty(_lib.mla_decode_workspace_size(p["cfg"], w.batch, w.n_q),
                         dtype=torch.uint8, device="cuda")
        _lib.mla_decode(p["cfg"], p["dw"].handle, p["q"], p["cache"], p["pt"], p["sl"], ref, ws)
        got = torch.full(shape, float("nan"), device="cuda")
        _lib.mla_decode_no_alloc(p["cfg"], p["dw"].handle, p["q"], p["cache"], p["pt"], p["sl"],
                                 got)
        torch.cuda.synchronize()
        _close(got.cpu().numpy(), ref.cpu().numpy(), w.dtype)
        if k == 0:
            first = got.cpu().numpy()
        elif k == len(problems):
            # the same problem gives the same bits, whatever came in between
            assert np.array_equal(got.cpu().numpy(), first)
    for p in problems:
        p["dw"].free()


def test_no_alloc_full_size_batch16():
    """The DeepSeek-V2-shape batch of 16 x 4096 cached tokens fits the array;
    two calls in a row match mla_decode."""
    w = synth.WORKLOADS["dsv2_b16_l4096"]
    cfg = config_for(w)
    need = _lib.mla_decode_workspace_size(cfg, w.batch, w.n_q)
    assert need <= _lib.MLA_NO_ALLOC_WORKSPACE_BYTES
    lens = synth.seq_lens(w)
    dw = DeviceWeights(w, synth.weights(w), cfg)
    pt, nb = synth.page_table(w, lens)
    store, _ = synth.fill_paged_cache(w, lens, pt, nb)
    _, qs = synth.queries(w)
    cache, ptd = to_device(store, w.dtype), to_device(pt, "i32")
    sl, q = to_device(lens, "i32"), to_device(qs, w.dtype)
    shape = (w.batch, w.n_q, w.n_h, w.d_v)
    ref = torch.full(shape, float("nan"), device="cuda")
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    _lib.mla_decode(cfg, dw.handle, q, cache, ptd, sl, ref, ws)
    for _ in range(2):
        got = torch.full(shape, float("nan"), device="cuda")
        _lib.mla_decode_no_alloc(cfg, dw.handle, q, cache, ptd, sl, got)
        torch.cuda.synchronize()
        _close(got.cpu().numpy(), ref.cpu().numpy(), w.dtype)
    dw.free()


def test_no_alloc_fits_by_workload():
    """Which of the benchmark workloads fit the fixed array: the fp32 tiny
    one, DeepSeek-V2 batch 16 and batch 4 x 131072 (2 queries) do; batch 64
    ragged and the 16-head batch of 256 need more scratch than the array
    holds and get MLA_ERR_WORKSPACE from mla_decode_no_alloc."""
    fits = {}
    for name in synth.WORKLOAD_ORDER:
        w = synth.WORKLOADS[name]
        need = _lib.mla_decode_workspace_size(config_for(w), w.batch, w.n_q)
        fits[name] = need <= _lib.MLA_NO_ALLOC_WORKSPACE_BYTES
        print(f"{name}: decode workspace {need} B ({need / 2**20:.2f} MiB), fits: {fits[name]}")
    assert fits["tiny_fp32"] and fits["dsv2_b16_l4096"]


def test_no_alloc_rejects_requests_larger_than_its_array():
    cfg = _lib.make_config(128, 5120, 512, 64, 128, 128)
    B, n_q = 1024, 1  # the absorbed queries alone need 144 MiB
    assert _lib.mla_decode_workspace_size(cfg, B, n_q) > _lib.MLA_NO_ALLOC_WORKSPACE_BYTES
    out = torch.full((4,), 3.0, device="cuda")
    st = _lib.load().mla_decode_no_alloc(ctypes.byref(cfg), None, None, None, 1, None, 1, None, B,
                                         n_q, ctypes.c_void_p(out.data_ptr()), None)
    assert st == 5  # MLA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(out == 3.0)
