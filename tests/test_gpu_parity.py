"""GPU parity: libmla (through its C ABI) against the fp64 oracle.

Tolerances:
  * fp32 workloads: max-abs <= 1e-4.
  * bf16 workloads: rel-L2 <= 5e-3 and max-abs <= 2e-2.
  * Cache placement and page tables: bit-exact.

Every input comes from the seeded generator. No expected value comes from
the CUDA path.
"""
import dataclasses
import math

import numpy as np
import pytest

from mla_latent_kv_73_b300 import _lib, synth
from mla_latent_kv_73_b300.device_inputs import (DeviceWeights, config_for, to_device,
                                                to_host_f32)
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


def check_bf16(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    mab = np.max(np.abs(got - ref))
    assert rel <= 5e-3 and mab <= 2e-2, f"{what}: rel-L2 {rel:.3e} max-abs {mab:.3e}"
    return rel, mab


def check_bf16_each(got, ref, what=""):
    """The bf16 bound applied to every sampled output vector on its own, so
    that one bad head cannot hide inside a pooled norm. Returns the worst
    rel-L2."""
    worst = 0.0
    for k, (g, r) in enumerate(zip(got, ref)):
        rel, _ = check_bf16(g, r, f"{what} sample {k}")
        worst = max(worst, rel)
    return worst


def check_f32(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    mab = np.max(np.abs(got - np.asarray(ref, dtype=np.float64)))
    assert np.isfinite(mab) and mab <= 1e-4, f"{what}: max-abs {mab:.3e}"
    return mab


def check(dtype, got, ref, what=""):
    return check_f32(got, ref, what) if dtype == "f32" else check_bf16(got, ref, what)


def small_workload(n_h=128, d_model=64, lens=(1, 64, 65, 200), n_q=1, dtype="bf16", seed=11,
                   d_c=512, d_r=64, d_nope=128, d_v=128):
    w = synth.Workload(f"small_{n_h}_{n_q}_{seed}", n_h=n_h, d_model=d_model, d_c=d_c, d_r=d_r,
                       d_nope=d_nope, d_v=d_v, batch=len(lens), n_q=n_q, len_lo=0, len_hi=0,
                       dtype=dtype, seed=seed)
    return w, np.asarray(lens, dtype=np.int32)


class Run:
    """One decode problem on the device: inputs, weights, workspace, output."""

    def __init__(self, w, lens, impl, fill=float("nan"), spare_blocks=3, q_mul=1.0):
        self.w, self.lens = w, lens
        self.cfg = config_for(w, impl)
        self.wts = synth.weights(w)
        self.dw = DeviceWeights(w, self.wts, self.cfg)
        pt, nb = synth.page_table(w, lens, spare_blocks=spare_blocks)
        self.pt_np, self.num_blocks = pt, nb
        store, self.rows = synth.fill_paged_cache(w, lens, pt, nb, fill_value=fill)
        self.cache = to_device(store, w.dtype)
        self.pt = to_device(pt, "i32")
        self.sl = to_device(lens.astype(np.int32), "i32")
        qv, qs = synth.queries(w)
        if q_mul != 1.0:
            # a power of two keeps every value exact in the workload's dtype
            assert math.frexp(q_mul)[0] == 0.5
            qv, qs = synth.to_dtype(qv * np.float32(q_mul), w.dtype)
        self.q_vals = qv
        self.q = to_device(qs, w.dtype)
        self.out = torch.full((w.batch, w.n_q, w.n_h, w.d_v), float("nan"), device="cuda")
        nbytes = _lib.mla_decode_workspace_size(self.cfg, w.batch, w.n_q, int(lens.sum()))
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")

    def decode(self):
        _lib.mla_decode(self.cfg, self.dw.handle, self.q, self.cache, self.pt, self.sl, self.out,
                        self.ws)
        torch.cuda.synchronize()
        return self.out.cpu().numpy()

    def oracle(self, samples=None):
        w = self.w
        return O.decode_materialised(self.q_vals, self.rows, self.lens, self.wts.W_uk,
                                     self.wts.W_uv, w.d_c, w.d_nope, w.d_v, w.scale,
                                     w.rope_base, samples=samples)


# ---------------------------------------------------------------------------
# a1: compress and append
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("wname,T", [("tiny_fp32", 5), ("tiny_fp32", 77),
                                     ("dsv2_b16_l4096", 16), ("dsv2_b16_l4096", 70),
                                     ("nh16_b256_ragged", 3)])
def test_append_places_rows_exactly(wname, T):
    w = synth.WORKLOADS[wname]
    B = 3
    lens = np.array([130, 64, 200], dtype=np.int32)
    pt, nb = synth.page_table(w, lens, spare_blocks=2)
    g = np.random.default_rng(5)
    # distinct (seq, pos) targets inside each sequence's pages
    pairs = set()
    while len(pairs) < T:
        b = int(g.integers(0, B))
        pairs.add((b, int(g.integers(0, lens[b]))))
    pairs = sorted(pairs, key=lambda _: g.random())
    seq_idx = np.array([p[0] for p in pairs], dtype=np.int32)
    pos = np.array([p[1] for p in pairs], dtype=np.int32)
    xv, xs = synth.hidden_states(w, T)
    wts = synth.weights(w)
    cfg = config_for(w)
    dw = DeviceWeights(w, wts, cfg)
    canary = 7.0
    cache = torch.full((nb, w.block_size, w.R), canary, device="cuda",
                       dtype=torch.float32 if w.dtype == "f32" else torch.bfloat16)
    _lib.mla_append_kv(cfg, dw.handle, to_device(xs, w.dtype), to_device(seq_idx, "i32"),
                       to_device(pos, "i32"), to_device(pt, "i32"), cache)
    torch.cuda.synchronize()
    st, code = _lib.mla_get_last_device_error()
    assert code == 0
    got = to_host_f32(cache).reshape(-1, w.R)
    rows = O.latent_rows(xv, wts.W_dkv, wts.W_kr, pos, w.rope_base)
    written = np.zeros(got.shape[0], dtype=bool)
    for t in range(T):
        r = O.paged_row_index(pt, seq_idx[t], pos[t], w.block_size)
        written[r] = True
        check(w.dtype, got[r], rows[t], f"row {t}")
    # every other row is bit-identical to the canary
    assert np.all(got[~written] == canary)
    dw.free()


@pytest.mark.parametrize("wname,T,d_model", [("dsv2_b16_l4096", 1024, None),
                                             ("dsv2_b16_l4096", 200, None),
                                             ("nh16_b256_ragged", 300, None),
                                             ("tiny_fp32", 600, None),
                                             ("tiny_fp32", 20, 4096)])
def test_append_bulk_and_far_positions(wname, T, d_model):
    """One call with many new tokens (the tile-GEMM path: 1024 and 300
    tokens, and 200 at d_model 5120, where the split-K kernel's staging does
    not fit; the last tile of 128 tokens partly filled), or a wide fp32
    model with few tokens (the direct-load path), at positions up to 131071:
    each row against the oracle's latent_rows (RoPE at the largest
    positions included), placed exactly, every other row untouched."""
    w = synth.WORKLOADS[wname]
    if d_model is not None:
        w = dataclasses.replace(w, d_model=d_model, name=f"{wname}_dm{d_model}")
    lens = np.array([131072, 70001, 3000], dtype=np.int32)
    pt, nb = synth.page_table(w, lens, spare_blocks=2)
    g = np.random.default_rng(31)
    pairs = {(0, 131071), (0, 131070), (1, 70000), (2, 0), (2, 2999)}
    while len(pairs) < T:
        b = int(g.integers(0, 3))
        pairs.add((b, int(g.integers(0, lens[b]))))
    pairs = sorted(pairs, key=lambda _: g.random())
    seq_idx = np.array([p[0] for p in pairs], dtype=np.int32)
    pos = np.array([p[1] for p in pairs], dtype=np.int32)
    xv, xs = synth.hidden_states(w, T, stream=3)
    wts = synth.weights(w)
    cfg = config_for(w)
    dw = DeviceWeights(w, wts, cfg)
    canary = 7.0
    cache = torch.full((nb, w.block_size, w.R), canary, device="cuda",
                       dtype=torch.float32 if w.dtype == "f32" else torch.bfloat16)
    _lib.mla_append_kv(cfg, dw.handle, to_device(xs, w.dtype), to_device(seq_idx, "i32"),
                       to_device(pos, "i32"), to_device(pt, "i32"), cache)
    torch.cuda.synchronize()
    st, code = _lib.mla_get_last_device_error()
    assert code == 0
    flat = cache.view(-1, w.R)
    # placement: exactly the T target rows differ from the canary
    changed = torch.nonzero(torch.any(flat != canary, dim=1)).flatten().cpu().numpy()
    want = np.array(sorted(O.paged_row_index(pt, seq_idx[t], pos[t], w.block_size)
                           for t in range(T)))
    assert np.array_equal(np.sort(changed), want)
    idx = torch.from_numpy(np.array([O.paged_row_index(pt, seq_idx[t], pos[t], w.block_size)
                                     for t in range(T)], dtype=np.int64)).cuda()
    got = to_host_f32(flat.index_select(0, idx))
    rows = O.latent_rows(xv, wts.W_dkv, wts.W_kr, pos, w.rope_base)
    for t in range(T):
        check(w.dtype, got[t], rows[t], f"row {t} (seq {seq_idx[t]}, pos {pos[t]})")
    dw.free()


def test_append_bad_indices_are_flagged_and_skipped():
    w = synth.WORKLOADS["tiny_fp32"]
    lens = np.array([64, 64], dtype=np.int32)
    pt, nb = synth.page_table(w, lens)
    pt[1, 0] = nb + 5  # page id out of range
    wts = synth.weights(w)
    cfg = config_for(w)
    dw = DeviceWeights(w, wts, cfg)
    xv, xs = synth.hidden_states(w, 3)
    cache = torch.zeros((nb, w.block_size, w.R), device="cuda")
    seq_idx = np.array([0, 5, 1], dtype=np.int32)   # 5: no such sequence
    pos = np.array([3, 0, 2], dtype=np.int32)       # token 2 hits the bad page
    _lib.mla_append_kv(cfg, dw.handle, to_device(xs, "f32"), to_device(seq_idx, "i32"),
                       to_device(pos, "i32"), to_device(pt, "i32"), cache)
    st, code = _lib.mla_get_last_device_error()
    assert code == (_lib.MLA_DEVERR_APPEND_INDEX | _lib.MLA_DEVERR_PAGE_RANGE)
    assert st == 7  # MLA_ERR_DEVICE_CHECK
    got = cache.cpu().numpy().reshape(-1, w.R)
    r0 = O.paged_row_index(pt, 0, 3, w.block_size)
    assert np.count_nonzero(np.any(got != 0, axis=1)) == 1 and np.any(got[r0] != 0)
    dw.free()


# ---------------------------------------------------------------------------
# a2..a5: decode
# ---------------------------------------------------------------------------


def test_tiny_fp32_end_to_end():
    """The fp32 workload: rows come from mla_append_kv, queries from the
    generator; compare with the oracle's own rows and decode."""
    w = synth.WORKLOADS["tiny_fp32"]
    lens = synth.seq_lens(w)
    cfg = config_for(w)
    assert _lib.mla_decode_impl(cfg) == _lib.MLA_IMPL_CUDA_CORE
    wts = synth.weights(w)
    dw = DeviceWeights(w, wts, cfg)
    pt, nb = synth.page_table(w, lens)
    T = int(lens.sum())
    xv, xs = synth.hidden_states(w, T)
    seq_idx = np.repeat(np.arange(w.batch), lens).astype(np.int32)
    pos = np.concatenate([np.arange(L) for L in lens]).astype(np.int32)
    cache = torch.zeros((nb, w.block_size, w.R), device="cuda")
    _lib.mla_append_kv(cfg, dw.handle, to_device(xs, "f32"), to_device(seq_idx, "i32"),
                       to_device(pos, "i32"), to_device(pt, "i32"), cache)
    qv, qs = synth.queries(w)
    out = torch.zeros((w.batch, w.n_q, w.n_h, w.d_v), device="cuda")
    ws = torch.empty(_lib.mla_decode_workspace_size(cfg, w.batch, w.n_q), dtype=torch.uint8,
                     device="cuda")
    _lib.mla_decode(cfg, dw.handle, to_device(qs, "f32"), cache, to_device(pt, "i32"),
                    to_device(lens, "i32"), out, ws)
    torch.cuda.synchronize()
    rows_all = O.latent_rows(xv, wts.W_dkv, wts.W_kr, pos, w.rope_base)
    seq_rows = [rows_all[seq_idx == b] for b in range(w.batch)]
    ref = O.decode_materialised(qv, seq_rows, lens, wts.W_uk, wts.W_uv, w.d_c, w.d_nope, w.d_v,
                                w.scale, w.rope_base)
    check_f32(out.cpu().numpy(), ref, "tiny fp32 end to end")
    # the tensor-core kernel does not take fp32
    cfg_tc = config_for(w, _lib.MLA_IMPL_TENSOR_CORE)
    with pytest.raises(_lib.MlaError) as ei:
        _lib.mla_decode(cfg_tc, dw.handle, to_device(qs, "f32"), cache, to_device(pt, "i32"),
                        to_device(lens, "i32"), out, ws)
    assert ei.value.status == 4  # MLA_ERR_UNSUPPORTED
    dw.free()


SMALL_CASES = {
    "ragged_nq1": dict(lens=(1, 64, 65, 200, 300)),
    "causal_nq2": dict(lens=(2, 65, 129, 640), n_q=2),
    "nh16": dict(n_h=16, lens=(1, 17, 64, 100, 129, 250, 333, 400, 3)),
    "one_long_seq": dict(lens=(64 * 37 + 5,)),
    "nh8_nq3": dict(n_h=8, n_q=3, lens=(3, 70, 191)),
}


@pytest.mark.parametrize("impl", list(IMPLS))
@pytest.mark.parametrize("case", list(SMALL_CASES))
def test_decode_small_bf16(impl, case):
    w, lens = small_workload(**SMALL_CASES[case])
    r = Run(w, lens, IMPLS[impl])
    got = r.decode()
    ref = r.oracle()
    check_bf16(got, ref, f"{case}/{impl}")
    r.dw.free()


def test_decode_small_fp32_shapes():
    w, lens = small_workload(n_h=4, d_model=32, d_c=32, d_r=8, d_nope=16, d_v=16,
                             lens=(2, 5, 64, 65, 130), n_q=2, dtype="f32")
    r = Run(w, lens, _lib.MLA_IMPL_AUTO)
    check_f32(r.decode(), r.oracle(), "small fp32")
    r.dw.free()


def test_decode_widest_heads_fp32():
    """d_nope = 800 (the query absorption stages 51 KB of queries in shared
    memory) and d_v = 1024, the widest head the config accepts."""
    w, lens = small_workload(n_h=2, d_model=32, d_c=32, d_r=8, d_nope=800, d_v=1024,
                             lens=(3, 70), n_q=1, dtype="f32")
    r = Run(w, lens, _lib.MLA_IMPL_AUTO)
    check_f32(r.decode(), r.oracle(), "widest heads fp32")
    r.dw.free()


def test_kernels_agree_and_steps_equal_fused():
    w, lens = small_workload(lens=(5, 128, 129, 700), n_q=2, seed=3)
    a = Run(w, lens, _lib.MLA_IMPL_TENSOR_CORE)
    out_tc = a.decode()
    out_tc2 = a.decode()
    assert np.array_equal(out_tc, out_tc2), "decode is not deterministic"
    # the three stage calls reproduce the fused call bit for bit
    out2 = torch.full_like(a.out, float("nan"))
    _lib.mla_decode_absorb_q(a.cfg, a.dw.handle, a.q, a.sl, a.pt.shape[1], a.ws)
    _lib.mla_decode_attend(a.cfg, a.cache, a.pt, a.sl, w.batch, w.n_q, a.ws)
    _lib.mla_decode_combine(a.cfg, a.dw.handle, a.sl, w.batch, w.n_q, out2, a.ws)
    torch.cuda.synchronize()
    assert np.array_equal(out2.cpu().numpy(), out_tc)
    b = Run(w, lens, _lib.MLA_IMPL_CUDA_CORE)
    check_bf16(b.decode(), out_tc, "cuda-core vs tensor-core")
    a.dw.free()
    b.dw.free()


def test_output_off_its_16_byte_alignment():
    """out at a 4-byte offset: the tensor-core combine writes 16-byte
    vectors, so the library takes the CUDA-core combine for it; the result
    matches the aligned call's within the bf16 bound."""
    w, lens = small_workload(lens=(5, 128, 129, 300), n_q=2, seed=4)
    r = Run(w, lens, _lib.MLA_IMPL_TENSOR_CORE)
    ref = r.decode()
    n = w.batch * w.n_q * w.n_h * w.d_v
    buf = torch.full((n + 1,), float("nan"), device="cuda")
    out = buf[1:].view(w.batch, w.n_q, w.n_h, w.d_v)
    assert out.data_ptr() % 16 == 4
    _lib.mla_decode(r.cfg, r.dw.handle, r.q, r.cache, r.pt, r.sl, out, r.ws)
    torch.cuda.synchronize()
    check_bf16(out.cpu().numpy(), ref, "misaligned out")
    check_bf16(out.cpu().numpy(), r.oracle(), "misaligned out vs oracle")
    r.dw.free()


def test_bad_lengths_and_pages_are_flagged():
    w, lens = small_workload(lens=(0, 70, 100))  # seq 0 shorter than n_q
    r = Run(w, lens, _lib.MLA_IMPL_TENSOR_CORE)
    got = r.decode()
    st, code = _lib.mla_get_last_device_error()
    assert code == _lib.MLA_DEVERR_SEQ_LEN
    assert np.all(got[0] == 0.0)
    ref = r.oracle(samples=[(b, 0, h) for b in (1, 2) for h in range(w.n_h)])
    check_bf16(np.array([got[b, 0, h] for (b, _, h) in ref]), np.array(list(ref.values())))
    # a page id outside the cache
    pt = r.pt_np.copy()
    pt[2, 0] = r.num_blocks + 1
    r.pt = to_device(pt, "i32")
    r.decode()
    st, code = _lib.mla_get_last_device_error()
    assert code & _lib.MLA_DEVERR_PAGE_RANGE
    r.dw.free()


def test_host_argument_checks():
    w, lens = small_workload(lens=(10, 20))
    r = Run(w, lens, _lib.MLA_IMPL_AUTO)
    small = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(_lib.MlaError) as ei:
        _lib.mla_decode(r.cfg, r.dw.handle, r.q, r.cache, r.pt, r.sl, r.out, small)
    assert ei.value.status == 5  # MLA_ERR_WORKSPACE
    mis = r.ws[1:]
    with pytest.raises(_lib.MlaError) as ei:
        _lib.mla_decode(r.cfg, r.dw.handle, r.q, r.cache, r.pt, r.sl, r.out, mis)
    assert ei.value.status == 5
    bad = config_for(w)
    bad.d_r = 3
    with pytest.raises(_lib.MlaError) as ei:
        _lib.mla_decode(bad, r.dw.handle, r.q, r.cache, r.pt, r.sl, r.out, r.ws)
    assert ei.value.status == 2  # MLA_ERR_SHAPE
    r.dw.free()


# ---------------------------------------------------------------------------
# Full-size workloads: sampled outputs against the oracle
# ---------------------------------------------------------------------------


def _samples(w, lens, g):
    bs = {int(np.argmin(lens)), int(np.argmax(lens))} | {int(x) for x in g.integers(0, w.batch, 2)}
    hs = {0, w.n_h - 1, int(g.integers(0, w.n_h))}
    return [(b, i, h) for b in sorted(bs) for i in sorted({0, w.n_q - 1}) for h in sorted(hs)][:16]


@pytest.mark.parametrize("wname", ["dsv2_b16_l4096", "dsv2_b64_ragged", "dsv2_b4_l131072_nq2",
                                   "nh16_b256_ragged"])
def test_full_size_sampled(wname):
    w = synth.WORKLOADS[wname]
    lens = synth.seq_lens(w)
    r = Run(w, lens, _lib.MLA_IMPL_AUTO, fill=0.0, spare_blocks=0)
    assert _lib.mla_decode_impl(r.cfg) == _lib.MLA_IMPL_TENSOR_CORE
    got = r.decode()
    assert np.all(np.isfinite(got))
    st, code = _lib.mla_get_last_device_error()
    assert code == 0
    samples = _samples(w, lens, np.random.default_rng(w.seed))
    ref = r.oracle(samples=samples)
    check_bf16_each([got[s] for s in samples], [ref[s] for s in samples], wname)
    r.dw.free()


# ---------------------------------------------------------------------------
# The attention core alone (a3 + a4): mla_decode_latent
# ---------------------------------------------------------------------------


def run_latent(r):
    """mla_decode_latent on Run r's cache with the seeded latent queries:
    (o_lat on the host, the query values the oracle takes)."""
    w = r.w
    qv, qs = synth.latent_queries(w)
    o = torch.full((w.batch, w.n_q, w.n_h, w.d_c), float("nan"), device="cuda")
    _lib.mla_decode_latent(r.cfg, to_device(qs, w.dtype), r.cache, r.pt, r.sl, o, r.ws)
    torch.cuda.synchronize()
    st, code = _lib.mla_get_last_device_error()
    assert code == 0
    return o.cpu().numpy(), qv


@pytest.mark.parametrize("impl", list(IMPLS))
@pytest.mark.parametrize("n_q", [1, 2])
def test_decode_latent_core_small(impl, n_q):
    """o_lat against the oracle's latent core, every (sequence, query, head)
    vector on its own; sequences of 2 to 700 tokens (ragged last pages)."""
    w, lens = small_workload(lens=(2, 64, 65, 200, 700), n_q=n_q, seed=61)
    r = Run(w, lens, IMPLS[impl])
    got, qv = run_latent(r)
    ref = O.decode_latent(qv, r.rows, lens, w.d_c, w.scale)
    keys = [(b, i, h) for b in range(w.batch) for i in range(n_q) for h in range(w.n_h)]
    check_bf16_each([got[k] for k in keys], [ref[k] for k in keys], f"latent {impl} n_q={n_q}")
    r.dw.free()


def test_decode_latent_core_unaligned_buffers():
    """q_abs one element off its 16-byte alignment: the query copy takes
    scalar loads and the result matches the oracle as the aligned call does.
    An o_lat off its 16-byte alignment is refused on the host (both merge
    kernels store 16-byte vectors), with nothing queued."""
    w, lens = small_workload(lens=(3, 100, 129), n_q=2, seed=62)
    r = Run(w, lens, _lib.MLA_IMPL_TENSOR_CORE)
    qv, qs = synth.latent_queries(w)
    qd = to_device(qs, w.dtype)
    qbuf = torch.empty(qd.numel() + 1, dtype=qd.dtype, device="cuda")
    qbuf[1:].copy_(qd.reshape(-1))
    q_off = qbuf[1:].view(qd.shape)
    assert q_off.data_ptr() % 16 != 0
    o = torch.full((w.batch, w.n_q, w.n_h, w.d_c), float("nan"), device="cuda")
    _lib.mla_decode_latent(r.cfg, q_off, r.cache, r.pt, r.sl, o, r.ws)
    torch.cuda.synchronize()
    st, code = _lib.mla_get_last_device_error()
    assert code == 0
    got = o.cpu().numpy()
    ref = O.decode_latent(qv, r.rows, lens, w.d_c, w.scale)
    keys = [(b, i, h) for b in range(w.batch) for i in range(w.n_q) for h in range(w.n_h)]
    check_bf16_each([got[k] for k in keys], [ref[k] for k in keys], "latent unaligned q")
    obuf = torch.zeros(o.numel() + 1, device="cuda")
    o_off = obuf[1:].view(o.shape)
    with pytest.raises(_lib.MlaError) as ei:
        _lib.mla_decode_latent(r.cfg, q_off, r.cache, r.pt, r.sl, o_off, r.ws)
    assert ei.value.status == 1  # MLA_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.all(obuf == 0)
    r.dw.free()


def test_decode_latent_core_fp32():
    w = synth.WORKLOADS["tiny_fp32"]
    lens = synth.seq_lens(w)
    r = Run(w, lens, _lib.MLA_IMPL_AUTO)
    got, qv = run_latent(r)
    check_f32(got, O.decode_latent(qv, r.rows, lens, w.d_c, w.scale), "latent fp32")
    r.dw.free()


def test_decode_latent_core_full_size_sampled():
    """The headline workload (batch 64, 512-32768 cached tokens) on the
    tensor-core attention: sampled o_lat vectors against the oracle."""
    w = synth.WORKLOADS["dsv2_b64_ragged"]
    lens = synth.seq_lens(w)
    r = Run(w, lens, _lib.MLA_IMPL_AUTO, fill=0.0, spare_blocks=0)
    got, qv = run_latent(r)
    assert np.all(np.isfinite(got))
    samples = _samples(w, lens, np.random.default_rng(w.seed + 7))
    ref = O.decode_latent(qv, r.rows, lens, w.d_c, w.scale, samples=samples)
    check_bf16_each([got[s] for s in samples], [ref[s] for s in samples], "latent b64")
    r.dw.free()


U_BF16 = 2.0 ** -8  # unit roundoff of bf16 (8 significant bits)


@pytest.mark.parametrize("impl", ["cuda_core", "tensor_core"])
@pytest.mark.parametrize("wname", ["dsv2_b16_l4096", "dsv2_b4_l131072_nq2"])
def test_full_size_peaked_softmax(wname, impl):
    """Queries scaled by 8: the scaled logits have a standard deviation of
    sigma = 8 instead of 1 (the workloads draw q, c and k_rope as N(0, 1), so
    q_lat . c + q_pe . k_rope has variance d_nope + d_r), and a few keys carry
    most of each softmax, as in a trained model. Every sampled vector is
    checked on its own.

    The CUDA-core attention keeps the absorbed query and every score in fp32:
    it meets the workloads' bound (rel-L2 5e-3, max-abs 2e-2).

    The tensor-core attention multiplies bf16 operands: rounding q_lat and
    q_pe to bf16 moves every score by up to u = 2^-8 of its terms, so the
    logits carry an error of order u * sigma and the softmax passes it on to
    the output at that relative size (the fp16 partial-score exchange adds
    2^-11 * sigma, the bf16 P 2^-8). At the workloads' sigma = 1 that is
    inside 5e-3; here the bound is r = u * sigma = 2^-5 on rel-L2 and 4r on
    max-abs (the workloads' pair has the same ratio)."""
    w = synth.WORKLOADS[wname]
    lens = synth.seq_lens(w)
    q_mul = 8.0
    r = Run(w, lens, IMPLS[impl], fill=0.0, spare_blocks=0, q_mul=q_mul)
    got = r.decode()
    st, code = _lib.mla_get_last_device_error()
    assert code == 0
    samples = _samples(w, lens, np.random.default_rng(w.seed + 100))
    ref = r.oracle(samples=samples)
    what = f"{wname} x8 {impl}"
    if impl == "cuda_core":
        check_bf16_each([got[s] for s in samples], [ref[s] for s in samples], what)
    else:
        bound = U_BF16 * q_mul
        for k, s_ in enumerate(samples):
            g_, r_ = np.asarray(got[s_], np.float64), np.asarray(ref[s_], np.float64)
            rel = np.linalg.norm(g_ - r_) / np.linalg.norm(r_)
            mab = np.max(np.abs(g_ - r_))
            assert np.all(np.isfinite(g_)) and rel <= bound and mab <= 4 * bound, \
                f"{what} sample {k}: rel-L2 {rel:.3e} max-abs {mab:.3e} (bound {bound:.3e})"
    r.dw.free()


# ---------------------------------------------------------------------------
# Prefill chunks: many new tokens per sequence in one call
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("impl", list(IMPLS))
@pytest.mark.parametrize("n_q", [64, 512])
def test_prefill_chunk_end_to_end(n_q, impl):
    """A prefill step: a chunk of n_q new tokens per sequence is appended
    with one mla_append_kv call (their rows computed from hidden states) and
    all of them are decoded in one mla_decode call, each new token seeing the
    cached context and the chunk's tokens up to itself (causal inside the
    chunk). Sequence 0 has 1000 tokens of earlier context; sequence 1 starts
    from nothing, so its first new token sees only itself. Sampled outputs
    against the oracle, which computes the chunk's rows itself (rounded once
    to the cache dtype, as the cache stores them)."""
    w = synth.Workload(f"prefill_{n_q}", n_h=128, d_model=1024, d_c=512, d_r=64, d_nope=128,
                       d_v=128, batch=2, n_q=n_q, len_lo=0, len_hi=0, dtype="bf16", seed=40)
    lens = np.array([1000 + n_q, n_q], dtype=np.int32)
    cfg = config_for(w, IMPLS[impl])
    wts = synth.weights(w)
    dw = DeviceWeights(w, wts, cfg)
    pt, nb = synth.page_table(w, lens, spare_blocks=1)
    # earlier context of sequence 0: drawn rows; the chunk's rows come from append
    ctx = synth.sequence_rows(w, 0, 1000)
    store = np.full((nb * w.block_size, w.R), synth.round_bf16(np.float32([np.nan]))[1][0],
                    dtype=np.uint16)
    for j in range(1000):
        store[O.paged_row_index(pt, 0, j, w.block_size)] = ctx[1][j]
    cache = to_device(store.reshape(nb, w.block_size, w.R), "bf16")
    T = int(2 * n_q)
    xv, xs = synth.hidden_states(w, T, stream=7)
    seq_idx = np.repeat(np.arange(2), n_q).astype(np.int32)
    pos = np.concatenate([np.arange(L - n_q, L) for L in lens]).astype(np.int32)
    ptd = to_device(pt, "i32")
    _lib.mla_append_kv(cfg, dw.handle, to_device(xs, "bf16"), to_device(seq_idx, "i32"),
                       to_device(pos, "i32"), ptd, cache)
    qv, qs = synth.queries(w)
    out = torch.full((2, n_q, w.n_h, w.d_v), float("nan"), device="cuda")
    ws = torch.empty(_lib.mla_decode_workspace_size(cfg, 2, n_q), dtype=torch.uint8,
                     device="cuda")
    _lib.mla_decode(cfg, dw.handle, to_device(qs, "bf16"), cache, ptd, to_device(lens, "i32"),
                    out, ws)
    torch.cuda.synchronize()
    st, code = _lib.mla_get_last_device_error()
    assert code == 0
    got = out.cpu().numpy()
    assert np.all(np.isfinite(got))
    new_rows = O.latent_rows(xv, wts.W_dkv, wts.W_kr, pos, w.rope_base)
    new_rows = synth.round_bf16(new_rows.astype(np.float32))[0]
    seq_rows = [np.concatenate([ctx[0], new_rows[:n_q]]), new_rows[n_q:]]
    g = np.random.default_rng(n_q)
    samples = [(b, i, h) for b in (0, 1) for i in sorted({0, 1, n_q // 2, n_q - 1,
                                                          int(g.integers(0, n_q))})
               for h in (0, int(g.integers(0, w.n_h)))]
    ref = O.decode_materialised(qv, seq_rows, lens, wts.W_uk, wts.W_uv, w.d_c, w.d_nope, w.d_v,
                                w.scale, w.rope_base, samples=samples)
    check_bf16_each([got[s] for s in samples], [ref[s] for s in samples],
                    f"prefill n_q={n_q} {impl}")
    dw.free()
