"""GPU parity of the full-fold layer (mla_decode_full) against the fp64 oracle.

The oracle side is ``layer_output_materialised``: q = x_q W_q, every head's
keys and values materialised, y = concat_h(o_h) W_o. The library folds
W_abs = W_q W_uk^T and W_uv W_o at load and never forms q_nope, keys,
values or o_h.

Tolerances are those of the per-head decode: max-abs <= 1e-4 for fp32, and
rel-L2 <= 5e-3 with max-abs <= 2e-2 for bf16. In bf16 the projected query
is rounded to bf16 before the attention, as q_lat is on the per-head path;
the folded weights and both projections stay in fp32.
"""
import numpy as np
import pytest

from mla_latent_kv_73_b300 import _lib, synth
from mla_latent_kv_73_b300.device_inputs import config_for, to_device
from oracle import mla_oracle as O

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

IMPLS = {"cuda_core": _lib.MLA_IMPL_CUDA_CORE, "tensor_core": _lib.MLA_IMPL_TENSOR_CORE}


@pytest.fixture(scope="module", autouse=True)
def _gpu(lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    st, code = _lib.mla_get_last_device_error()
    assert code == 0, f"device error word left set: {code:#x}"


def workload(n_h, d_model, d_c, d_r, d_nope, d_v, lens, n_q, dtype, seed):
    w = synth.Workload(f"full_{n_h}_{d_model}_{n_q}_{seed}", n_h=n_h, d_model=d_model, d_c=d_c,
                       d_r=d_r, d_nope=d_nope, d_v=d_v, batch=len(lens), n_q=n_q, len_lo=0,
                       len_hi=0, dtype=dtype, seed=seed)
    return w, np.asarray(lens, dtype=np.int32)


def check(dtype, got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    mab = np.max(np.abs(got - ref))
    if dtype == "f32":
        assert mab <= 1e-4, f"{what}: max-abs {mab:.3e}"
        return
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    assert rel <= 5e-3 and mab <= 2e-2, f"{what}: rel-L2 {rel:.3e} max-abs {mab:.3e}"


class FullRun:
    """One full-fold layer problem on the device."""

    def __init__(self, w, lens, impl=_lib.MLA_IMPL_AUTO, y_offset=0):
        self.w, self.lens = w, lens
        self.cfg = config_for(w, impl)
        self.wts = synth.weights(w)
        raw = {k: to_device(self.wts.raw[k], w.dtype) for k in ("W_q", "W_uk", "W_uv", "W_o")}
        self.fw = _lib.mla_fold_full(self.cfg, raw["W_q"], raw["W_uk"], raw["W_uv"], raw["W_o"])
        torch.cuda.synchronize()
        pt, nb = synth.page_table(w, lens, spare_blocks=2)
        store, self.rows = synth.fill_paged_cache(w, lens, pt, nb, fill_value=float("nan"))
        self.cache = to_device(store, w.dtype)
        self.pt = to_device(pt, "i32")
        self.sl = to_device(lens, "i32")
        B, n_q = len(lens), w.n_q
        xv, xs = synth.hidden_states(w, B * n_q, stream=1)
        self.x_vals = xv.reshape(B, n_q, w.d_model)
        self.x = to_device(xs.reshape(B, n_q, w.d_model), w.dtype)
        n = B * n_q * w.d_model
        self.y_buf = torch.full((n + y_offset,), float("nan"), device="cuda")
        self.y = self.y_buf[y_offset:].view(B, n_q, w.d_model)
        self.ws = torch.empty(_lib.mla_decode_full_workspace_size(self.cfg, B, n_q),
                              dtype=torch.uint8, device="cuda")

    def decode(self):
        _lib.mla_decode_full(self.cfg, self.fw, self.x, self.cache, self.pt, self.sl, self.y,
                             self.ws)
        torch.cuda.synchronize()
        return self.y.cpu().numpy()

    def oracle(self, tokens=None):
        w = self.w
        return O.layer_output_materialised(self.x_vals, self.rows, self.lens, self.wts.W_q,
                                           self.wts.W_uk, self.wts.W_uv, self.wts.W_o, w.d_c,
                                           w.d_nope, w.d_v, w.scale, w.rope_base, tokens=tokens)

    def free(self):
        _lib.mla_full_weights_free(self.fw)


@pytest.mark.parametrize("n_q", [1, 2])
def test_full_fold_tiny_fp32(n_q):
    w, lens = workload(4, 64, 32, 8, 16, 16, (2, 64, 65, 200), n_q, "f32", seed=21)
    r = FullRun(w, lens)
    check("f32", r.decode(), r.oracle(), "tiny fp32")
    r.free()


@pytest.mark.parametrize("impl", ["cuda_core", "tensor_core"])
@pytest.mark.parametrize("n_q", [1, 2])
def test_full_fold_bf16_dsv2_latent(impl, n_q):
    w, lens = workload(16, 256, 512, 64, 128, 128, (2, 64, 65, 200, 700), n_q, "bf16", seed=22)
    r = FullRun(w, lens, IMPLS[impl])
    check("bf16", r.decode(), r.oracle(), f"bf16 {impl}")
    r.free()


def test_full_fold_unaligned_output_written_directly():
    """n_h*d_c = 16 rows of W_vo are one K split, so the output projection
    writes y itself (no split partials), here at a 4-byte offset from a
    16-byte boundary."""
    w, lens = workload(2, 64, 8, 2, 4, 4, (3, 90), 1, "f32", seed=23)
    r = FullRun(w, lens, y_offset=1)
    assert r.y.data_ptr() % 16 == 4
    check("f32", r.decode(), r.oracle(), "unaligned y")
    assert torch.isnan(r.y_buf[0]).item()  # nothing written before y
    r.free()


def test_full_fold_sampled_wider_layer():
    """n_h = 16, d_model = 2048 (the small-head workload's widths), longer
    sequences, two query tokens, through the default kernel."""
    w, lens = workload(16, 2048, 512, 64, 128, 128, (1500, 333, 64), 2, "bf16", seed=24)
    r = FullRun(w, lens)
    got = r.decode()
    want = r.oracle()
    check("bf16", got, want, "wider layer")
    r.free()


def test_full_fold_deterministic_and_checks_workspace():
    w, lens = workload(16, 256, 512, 64, 128, 128, (2, 300, 129), 2, "bf16", seed=25)
    r = FullRun(w, lens)
    a = r.decode()
    b = r.decode()
    assert np.array_equal(a, b), "full-fold decode is not deterministic"
    small = r.ws[:64 * 1024]  # far below the partials alone
    with pytest.raises(_lib.MlaError) as e:
        _lib.mla_decode_full(r.cfg, r.fw, r.x, r.cache, r.pt, r.sl, r.y, small)
    assert e.value.status == 5  # MLA_ERR_WORKSPACE
    r.free()


def test_full_fold_rows_not_16_byte_aligned():
    """n_h*(d_c + d_r) = 114 and d_model = 70 are not multiples of 4 floats, so
    the bulk-copy ring cannot take the folded rows; the register form runs."""
    w, lens = workload(3, 70, 32, 6, 16, 16, (5, 77, 130), 2, "f32", seed=26)
    r = FullRun(w, lens)
    check("f32", r.decode(), r.oracle(), "unaligned rows")
    r.free()
