"""GPU parity of the fp8 (e4m3) latent cache against the fp64 oracle.

  * mla_quantize_rows_fp8: codes and row scales bit-exact against the
    oracle's quantize_rows_fp8 computed in fp32 (the precision the kernel
    takes its decisions in), placed exactly through the page table.
  * mla_append_kv_fp8: rows from hidden states; every dequantised row within
    the e4m3 rounding bound of the oracle's latent_rows, placement exact.
  * mla_decode_fp8: against decode_materialised over the dequantised rows
    (code * scale), with the bf16 workloads' tolerance (rel-L2 5e-3, max-abs
    2e-2), at small sizes and sampled at the four full-size workloads.

The cache codes of the decode tests are drawn directly as e4m3 bytes by the
seeded generator; the oracle decodes the same bytes.
"""
import numpy as np
import pytest

from mla_latent_kv_73_b300 import _lib, synth
from mla_latent_kv_73_b300.device_inputs import DeviceWeights, config_for, to_device
from oracle import mla_oracle as O

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu(lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    st, code = _lib.mla_get_last_device_error()
    assert code == 0, f"device error word left set: {code:#x}"


def e4m3_values(codes):
    """Values of e4m3 code bytes (a format decode by torch)."""
    c = torch.as_tensor(np.ascontiguousarray(codes, dtype=np.uint8))
    return c.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def check_bf16(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    mab = np.max(np.abs(got - ref))
    assert rel <= 5e-3 and mab <= 2e-2, f"{what}: rel-L2 {rel:.3e} max-abs {mab:.3e}"
    return rel


def small(n_h=128, lens=(1, 64, 65, 200), n_q=1, seed=51, d_model=64):
    w = synth.Workload(f"fp8_{n_h}_{n_q}_{seed}", n_h=n_h, d_model=d_model, d_c=512, d_r=64,
                       d_nope=128, d_v=128, batch=len(lens), n_q=n_q, len_lo=0, len_hi=0,
                       dtype="bf16", seed=seed)
    return w, np.asarray(lens, dtype=np.int32)


# ---------------------------------------------------------------------------
# quantiser and append
# ---------------------------------------------------------------------------


def test_quantize_rows_bit_exact_and_placed():
    w, _ = small(lens=(300, 100, 5))
    lens = np.array([300, 100, 5], dtype=np.int32)
    pt, nb = synth.page_table(w, lens, spare_blocks=2)
    g = np.random.default_rng(52)
    T = 257
    rows = (g.standard_normal((T, w.R)) * np.exp(g.uniform(-6, 6, (T, 1)))).astype(np.float32)
    rows[3] = 0.0                                   # a row of zeros: scale 1
    rows[4, :] = 1e-3                               # every element at the maximum
    rows[5] = g.uniform(-1, 1, w.R).astype(np.float32) * 2.0 ** -20  # tiny: subnormal codes
    rows[6, 7] = 1e4                                # one outlier dominates the scale
    pairs = set()
    while len(pairs) < T:
        b = int(g.integers(0, 3))
        pairs.add((b, int(g.integers(0, lens[b]))))
    pairs = sorted(pairs, key=lambda _: g.random())
    seq_idx = np.array([p[0] for p in pairs], dtype=np.int32)
    pos = np.array([p[1] for p in pairs], dtype=np.int32)
    cfg = config_for(w)
    canary_code, canary_scale = 0x5A, -7.0
    cache = torch.full((nb, w.block_size, w.R), canary_code, dtype=torch.uint8, device="cuda")
    scales = torch.full((nb, w.block_size), canary_scale, device="cuda")
    _lib.mla_quantize_rows_fp8(cfg, torch.from_numpy(rows).cuda(), to_device(seq_idx, "i32"),
                               to_device(pos, "i32"), to_device(pt, "i32"), cache, scales)
    torch.cuda.synchronize()
    st, code = _lib.mla_get_last_device_error()
    assert code == 0
    codes_ref, scales_ref = O.quantize_rows_fp8(rows, dtype=np.float32)
    flat_c = cache.view(-1, w.R).cpu().numpy()
    flat_s = scales.view(-1).cpu().numpy()
    idx = np.array([O.paged_row_index(pt, seq_idx[t], pos[t], w.block_size) for t in range(T)])
    got_vals = e4m3_values(flat_c[idx])
    assert np.array_equal(got_vals, codes_ref), "codes differ from the oracle's"
    assert np.array_equal(flat_s[idx].astype(np.float64), scales_ref), "scales differ"
    untouched = np.ones(flat_c.shape[0], dtype=bool)
    untouched[idx] = False
    assert np.all(flat_c[untouched] == canary_code) and np.all(flat_s[untouched] == canary_scale)


@pytest.mark.parametrize("T,d_model", [(70, 1024), (600, 1024), (300, 5120)])
def test_append_fp8_rows_within_the_rounding_bound(T, d_model):
    """Rows from hidden states (one chunk; three chunks of at most 256; at
    d_model 5120 a 256-token chunk on the tile GEMM and a 44-token one on
    the split-K kernel), dequantised, against the oracle's fp64 rows: each
    element within half an e4m3 step (2^-4 of its magnitude in the normal
    range, 2^-10 of the row scale below it), plus the fp32 row's own
    rounding."""
    w = synth.Workload("fp8_append", n_h=128, d_model=d_model, d_c=512, d_r=64, d_nope=128,
                       d_v=128, batch=3, n_q=1, len_lo=0, len_hi=0, dtype="bf16", seed=53)
    lens = np.array([131072, 900, 64], dtype=np.int32)
    pt, nb = synth.page_table(w, lens)
    g = np.random.default_rng(54)
    pairs = {(0, 131071), (0, 0)}
    while len(pairs) < T:
        b = int(g.integers(0, 3))
        pairs.add((b, int(g.integers(0, lens[b]))))
    pairs = sorted(pairs, key=lambda _: g.random())
    seq_idx = np.array([p[0] for p in pairs], dtype=np.int32)
    pos = np.array([p[1] for p in pairs], dtype=np.int32)
    xv, xs = synth.hidden_states(w, T, stream=9)
    wts = synth.weights(w)
    cfg = config_for(w)
    dw = DeviceWeights(w, wts, cfg)
    cache = torch.full((nb, w.block_size, w.R), 0x5A, dtype=torch.uint8, device="cuda")
    scales = torch.full((nb, w.block_size), -7.0, device="cuda")
    ws = torch.empty(_lib.mla_append_kv_fp8_workspace_size(cfg, T), dtype=torch.uint8,
                     device="cuda")
    _lib.mla_append_kv_fp8(cfg, dw.handle, to_device(xs, "bf16"), to_device(seq_idx, "i32"),
                           to_device(pos, "i32"), to_device(pt, "i32"), cache, scales, ws)
    torch.cuda.synchronize()
    st, code = _lib.mla_get_last_device_error()
    assert code == 0
    flat_c = cache.view(-1, w.R)
    flat_s = scales.view(-1)
    changed = torch.nonzero(flat_s != -7.0).flatten().cpu().numpy()
    idx = np.array([O.paged_row_index(pt, seq_idx[t], pos[t], w.block_size) for t in range(T)])
    assert np.array_equal(np.sort(changed), np.sort(idx))
    ti = torch.from_numpy(idx.astype(np.int64)).cuda()
    codes = e4m3_values(flat_c.index_select(0, ti).cpu().numpy())
    sc = flat_s.index_select(0, ti).cpu().numpy().astype(np.float64)
    deq = O.dequantize_rows_fp8(codes, sc)
    rows = O.latent_rows(xv, wts.W_dkv, wts.W_kr, pos, w.rope_base)
    amax = np.max(np.abs(rows), axis=1)
    assert np.allclose(sc, amax / 448.0, rtol=1e-5)
    u = np.abs(rows) / sc[:, None]
    bound = np.where(u >= 2.0 ** -6, 2.0 ** -4 * u, 2.0 ** -10) * sc[:, None]
    err = np.abs(deq - rows)
    assert np.all(err <= bound * 1.001 + 1e-5 * amax[:, None]), float(np.max(err / (bound + 1e-30)))
    dw.free()


# ---------------------------------------------------------------------------
# decode
# ---------------------------------------------------------------------------


class Fp8Run:
    """One decode problem over an fp8 cache: the codes of the sequences in
    ``keep`` (all if None) come from the generator; the other sequences'
    rows are random bytes drawn on the device (their outputs are not
    checked)."""

    def __init__(self, w, lens, keep=None, spare_blocks=2, uniform=False):
        self.w, self.lens = w, lens
        self.cfg = config_for(w)
        self.wts = synth.weights(w)
        self.dw = DeviceWeights(w, self.wts, self.cfg)
        pt, nb = synth.page_table(w, lens, spare_blocks=spare_blocks)
        self.pt_np, self.num_blocks = pt, nb
        bs = w.block_size
        gen = torch.Generator(device="cuda")
        gen.manual_seed(w.seed)
        # bytes 0..126 with a random sign bit: never the NaN patterns 0x7f, 0xff
        mag = torch.randint(0, 127, (nb, bs, w.R), generator=gen, device="cuda", dtype=torch.uint8)
        sgn = torch.randint(0, 2, (nb, bs, w.R), generator=gen, device="cuda", dtype=torch.uint8)
        self.cache = mag | (sgn << 7)
        del mag, sgn
        self.scales = torch.rand((nb, bs), generator=gen, device="cuda") * 0.01
        self.rows = [None] * len(lens)
        want = range(len(lens)) if keep is None else keep
        flat_c = self.cache.view(-1, w.R)
        flat_s = self.scales.view(-1)
        for b in want:
            gen_codes = synth.fp8_uniform_codes if uniform else synth.fp8_sequence_codes
            c, sc = gen_codes(w, b, lens[b])
            idx = np.array([O.paged_row_index(pt, b, j, bs) for j in range(int(lens[b]))])
            ti = torch.from_numpy(idx.astype(np.int64)).cuda()
            flat_c.index_copy_(0, ti, torch.from_numpy(c).cuda())
            flat_s.index_copy_(0, ti, torch.from_numpy(sc).cuda())
            self.rows[b] = O.dequantize_rows_fp8(e4m3_values(c), sc.astype(np.float64))
        self.pt = to_device(pt, "i32")
        self.sl = to_device(lens.astype(np.int32), "i32")
        qv, qs = synth.queries(w)
        self.q_vals = qv
        self.q = to_device(qs, "bf16")
        self.out = torch.full((w.batch, w.n_q, w.n_h, w.d_v), float("nan"), device="cuda")
        self.ws = torch.empty(_lib.mla_decode_workspace_size(self.cfg, w.batch, w.n_q),
                              dtype=torch.uint8, device="cuda")

    def decode(self):
        _lib.mla_decode_fp8(self.cfg, self.dw.handle, self.q, self.cache, self.scales, self.pt,
                            self.sl, self.out, self.ws)
        torch.cuda.synchronize()
        return self.out.cpu().numpy()

    def oracle(self, samples=None):
        w = self.w
        return O.decode_materialised(self.q_vals, self.rows, self.lens, self.wts.W_uk,
                                     self.wts.W_uv, w.d_c, w.d_nope, w.d_v, w.scale,
                                     w.rope_base, samples=samples)


SMALL = {
    "ragged_nq1": dict(lens=(1, 64, 65, 200, 300)),
    "causal_nq2": dict(lens=(2, 65, 129, 640), n_q=2),
    "nh16": dict(n_h=16, lens=(1, 17, 64, 100, 129, 250, 333, 400, 3)),
    "one_long_seq": dict(lens=(64 * 37 + 5,)),
    "all_codes": dict(lens=(3, 130, 700), uniform=True),
}


@pytest.mark.parametrize("case", list(SMALL))
def test_decode_fp8_small(case):
    kw = dict(SMALL[case])
    uniform = kw.pop("uniform", False)
    w, lens = small(**kw)
    r = Fp8Run(w, lens, uniform=uniform)
    got = r.decode()
    st, code = _lib.mla_get_last_device_error()
    assert code == 0
    ref = r.oracle()
    for b in range(w.batch):
        check_bf16(got[b], ref[b], f"{case} sequence {b}")
    # deterministic, call after call
    assert np.array_equal(r.decode(), got)
    r.dw.free()


def test_decode_fp8_rejects_what_it_cannot_run():
    w, lens = small(lens=(10, 20))
    r = Fp8Run(w, lens)
    bad = config_for(w, _lib.MLA_IMPL_CUDA_CORE)
    with pytest.raises(_lib.MlaError) as ei:
        _lib.mla_decode_fp8(bad, r.dw.handle, r.q, r.cache, r.scales, r.pt, r.sl, r.out, r.ws)
    assert ei.value.status == 4  # MLA_ERR_UNSUPPORTED
    with pytest.raises(_lib.MlaError) as ei:
        _lib.mla_decode_fp8(r.cfg, r.dw.handle, r.q, r.cache, r.scales.view(-1)[1:], r.pt, r.sl,
                            r.out, r.ws)
    assert ei.value.status == 1  # MLA_ERR_INVALID_ARG: row scales not 16-byte aligned
    r.dw.free()


def _samples(w, lens, g):
    bs = {int(np.argmin(lens)), int(np.argmax(lens))} | {int(x) for x in g.integers(0, w.batch, 2)}
    hs = {0, w.n_h - 1, int(g.integers(0, w.n_h))}
    return [(b, i, h) for b in sorted(bs) for i in sorted({0, w.n_q - 1}) for h in sorted(hs)][:16]


@pytest.mark.parametrize("wname", ["dsv2_b16_l4096", "dsv2_b64_ragged", "dsv2_b4_l131072_nq2",
                                   "nh16_b256_ragged"])
def test_decode_fp8_full_size_sampled(wname):
    w = synth.WORKLOADS[wname]
    lens = synth.seq_lens(w)
    samples = _samples(w, lens, np.random.default_rng(w.seed + 7))
    r = Fp8Run(w, lens, keep=sorted({b for b, _, _ in samples}), spare_blocks=0)
    got = r.decode()
    st, code = _lib.mla_get_last_device_error()
    assert code == 0
    ref = r.oracle(samples=samples)
    for k, s in enumerate(samples):
        check_bf16(got[s], ref[s], f"{wname} sample {k}")
    r.dw.free()
