"""GPU parity of one layer's decode step (mla_decode_layer) against the oracle.

The call appends the new tokens' rows from their hidden states, decodes
their queries and projects concat_h(o_h) through W_o. The oracle side:
the cache rows of the new tokens are the oracle's own latent rows rounded
once to the cache dtype (the other rows are the generated ones), then
``decode_materialised`` for `out` and ``layer_step_materialised`` for y.

Tolerances are those of the per-head decode: max-abs <= 1e-4 for fp32, and
rel-L2 <= 5e-3 with max-abs <= 2e-2 for bf16.
"""
import numpy as np
import pytest

from mla_latent_kv_73_b300 import _lib, synth
from mla_latent_kv_73_b300.device_inputs import DeviceWeights, config_for, to_device
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


def run_layer(n_h, d_model, d_c, d_r, d_nope, d_v, lens, n_q, dtype, seed,
              impl=_lib.MLA_IMPL_AUTO, w_o_offset=0, out_offset=0):
    w = synth.Workload(f"layer_{n_h}_{d_model}_{n_q}_{seed}", n_h=n_h, d_model=d_model, d_c=d_c,
                       d_r=d_r, d_nope=d_nope, d_v=d_v, batch=len(lens), n_q=n_q, len_lo=0,
                       len_hi=0, dtype=dtype, seed=seed)
    lens = np.asarray(lens, dtype=np.int32)
    B = len(lens)
    cfg = config_for(w, impl)
    wts = synth.weights(w)
    dw = DeviceWeights(w, wts, cfg)
    w_o = to_device(wts.raw["W_o"], dtype)
    if w_o_offset:  # the same matrix one element off its allocation's alignment
        buf = torch.empty(w_o.numel() + w_o_offset, dtype=w_o.dtype, device="cuda")
        buf[w_o_offset:].copy_(w_o.reshape(-1))
        w_o = buf[w_o_offset:].view(w_o.shape)
    pt, nb = synth.page_table(w, lens, spare_blocks=2)
    store, rows = synth.fill_paged_cache(w, lens, pt, nb, fill_value=float("nan"))
    cache = to_device(store, dtype)
    T = B * n_q
    xv, xs = synth.hidden_states(w, T, stream=2)
    seq_idx = np.repeat(np.arange(B), n_q).astype(np.int32)
    pos = np.concatenate([np.arange(L - n_q, L) for L in lens]).astype(np.int32)
    qv, qs = synth.queries(w)
    out = torch.full((B * n_q * n_h * d_v + out_offset,), float("nan"), device="cuda")
    out = out[out_offset:].view(B, n_q, n_h, d_v)  # off 16-byte alignment when out_offset % 4
    y = torch.full((B, n_q, d_model), float("nan"), device="cuda")
    ws = torch.empty(_lib.mla_decode_layer_workspace_size(cfg, B, n_q), dtype=torch.uint8,
                     device="cuda")
    _lib.mla_decode_layer(cfg, dw.handle, w_o, to_device(xs, dtype), to_device(seq_idx, "i32"),
                          to_device(pos, "i32"), to_device(qs, dtype), cache,
                          to_device(pt, "i32"), to_device(lens, "i32"), out, y, ws)
    torch.cuda.synchronize()
    # the oracle's rows: the new tokens' rows computed by the oracle, rounded
    # once to the cache dtype, in place of the generated ones
    new_rows = synth.to_dtype(O.latent_rows(xv, wts.W_dkv, wts.W_kr, pos, w.rope_base)
                              .astype(np.float32), dtype)[0]
    seq_rows = []
    for b in range(B):
        r = np.array(rows[b], dtype=np.float64, copy=True)
        r[lens[b] - n_q:] = new_rows[b * n_q:(b + 1) * n_q]
        seq_rows.append(r)
    o_ref = O.decode_materialised(qv, seq_rows, lens, wts.W_uk, wts.W_uv, d_c, d_nope, d_v,
                                  w.scale, w.rope_base)
    y_ref = O.layer_step_materialised(qv, seq_rows, lens, wts.W_uk, wts.W_uv, wts.W_o, d_c,
                                      d_nope, d_v, w.scale, w.rope_base)
    res = out.cpu().numpy(), y.cpu().numpy(), o_ref, y_ref
    dw.free()
    return res


@pytest.mark.parametrize("n_q", [1, 2])
def test_layer_tiny_fp32(n_q):
    out, y, o_ref, y_ref = run_layer(4, 64, 32, 8, 16, 16, (2, 64, 65, 200), n_q, "f32", 31)
    check("f32", out, o_ref, "out")
    check("f32", y, y_ref, "y")


@pytest.mark.parametrize("impl", ["cuda_core", "tensor_core"])
@pytest.mark.parametrize("n_q", [1, 2])
def test_layer_bf16_dsv2_latent(impl, n_q):
    out, y, o_ref, y_ref = run_layer(16, 256, 512, 64, 128, 128, (2, 64, 65, 200, 700), n_q,
                                     "bf16", 32, IMPLS[impl])
    check("bf16", out, o_ref, f"out {impl}")
    check("bf16", y, y_ref, f"y {impl}")


def test_layer_output_projection_register_form():
    """d_model = 260 bf16 rows are not 16-byte multiples, and W_o sits one
    element off its alignment: the projection takes scalar loads."""
    out, y, o_ref, y_ref = run_layer(16, 260, 512, 64, 128, 128, (3, 129), 1, "bf16", 33,
                                     w_o_offset=1)
    check("bf16", out, o_ref, "out")
    check("bf16", y, y_ref, "y")


def test_layer_dsv2_widths():
    """DeepSeek-V2 widths (n_h = 128, d_model = 5120): the W_o stream spans
    many K splits."""
    out, y, o_ref, y_ref = run_layer(128, 5120, 512, 64, 128, 128, (70, 257), 1, "bf16", 34)
    check("bf16", out, o_ref, "out")
    check("bf16", y, y_ref, "y")


@pytest.mark.parametrize("lens,n_q,d_model", [
    ((3, 64, 65, 130, 200, 257) * 4, 2, 200),  # 48 tokens; outputs 128..199 fill a tile partly
    ((7, 64, 129, 300) * 8, 2, 384),            # 64 tokens: the projection's widest token tile
    ((5, 90) * 20, 2, 256),                     # 80 tokens: past the tensor-core projection's 64
])
def test_layer_token_counts_and_ragged_outputs(lens, n_q, d_model):
    out, y, o_ref, y_ref = run_layer(16, d_model, 512, 64, 128, 128, lens, n_q, "bf16", 35)
    check("bf16", out, o_ref, "out")
    check("bf16", y, y_ref, "y")


def test_layer_projection_paths_agree():
    """out off its 16-byte alignment sends the step through the CUDA-core
    combine and projection (fp32 out); the aligned call goes through the
    tensor-core ones (out as a bf16 hi + lo pair). Both match the oracle, and
    each other to well within the bf16 bound."""
    args = (16, 512, 512, 64, 128, 128, (9, 64, 300), 2, "bf16", 36)
    out_a, y_a, o_ref, y_ref = run_layer(*args)
    out_b, y_b, _, _ = run_layer(*args, out_offset=1)
    check("bf16", y_a, y_ref, "y tensor-core projection")
    check("bf16", y_b, y_ref, "y CUDA-core projection")
    for a, b, what in ((out_a, out_b, "combines"), (y_a, y_b, "projections")):
        rel = np.linalg.norm(a - b) / np.linalg.norm(b)
        assert rel <= 1e-4, f"{what} differ: rel-L2 {rel:.3e}"
