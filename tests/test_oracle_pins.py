"""Pins for the fp64 oracle. CPU only.

Each test ties an oracle function to something the oracle does not compute
itself: a number printed on a page, a closed form, a library routine
(torch's scaled_dot_product_attention), an invariant of the mathematics, or a
brute-force construction. ``test_planted_mistakes_are_caught`` then plants
plausible bugs in the oracle and checks that these pins catch them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import mla_oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")
GiB = 1 << 30


def gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# Printed numbers: cache bytes, capacity, parameters, operation counts
# ---------------------------------------------------------------------------


def test_cache_bytes_printed_table():
    g = gold("p1_cache_bytes.json")
    for shape in g["shapes"].values():
        L, H, D = shape["layers"], shape["heads"], shape["head_dim"]
        mha = O.kv_cache_bytes(L, H, D, 1, shape["dtype_bytes"])
        gqa = O.kv_cache_bytes(L, 8, D, 1, shape["dtype_bytes"])
        mla = O.mla_cache_bytes(L, shape["d_c"], shape["d_rope"], 1, shape["dtype_bytes"])
        assert (mha, gqa, mla) == (shape["mha"], shape["gqa8"], shape["mla"])
        assert f"{mha / gqa:.1f}" == shape["gqa8_ratio"]
        assert f"{mha / mla:.1f}" == shape["mla_ratio"]
        assert f"{gqa / mla:.1f}" == shape["mla_vs_gqa8"]


def test_decoupled_rope_cost_printed():
    g = gold("p1_cache_bytes.json")["decoupled_rope_deepseek_v2"]
    latent = O.mla_cache_bytes(60, 512, 0, 1)
    full = O.mla_cache_bytes(60, 512, 64, 1)
    assert (latent, full, full - latent) == (g["latent_only"], g["with_rope"], g["added"])
    assert f"{100 * (full - latent) / latent:.1f}" == g["added_percent"]
    assert f"{O.kv_cache_bytes(60, 128, 128, 1) / full:.1f}" == g["vs_mha"]


def test_per_layer_elements_and_unverifiable_quote():
    g = gold("p1_cache_bytes.json")
    e = g["per_layer_elements"]
    assert O.mla_cache_bytes(1, 512, 64, 1, dtype_bytes=1) == e["mla"]
    assert O.kv_cache_bytes(1, 128, 128, 1, dtype_bytes=1) == e["mha"]
    # The quoted 93.3% is not what the pages' formulas give; record what they do give.
    red = 1 - O.mla_cache_bytes(60, 512, 64, 1) / O.kv_cache_bytes(60, 128, 128, 1)
    assert f"{100 * red:.2f}" == "98.24"
    assert g["quoted_not_derivable"]["reduction_vs_mha_percent_quoted"] == "93.3"


def test_capacity_in_80_gib_printed():
    g = gold("p1_capacity_80gib.json")
    s = g["shape"]
    budget = g["budget_gib"] * GiB
    for row in g["rows"]:
        n = row["context"]
        mha = O.kv_cache_bytes(s["layers"], s["heads"], s["head_dim"], n)
        gqa = O.kv_cache_bytes(s["layers"], s["gqa_groups"], s["head_dim"], n)
        mla = O.mla_cache_bytes(s["layers"], s["d_c"], s["d_rope"], n)
        assert f"{mha / GiB:.2f}" == row["mha_gib"]
        assert f"{gqa / GiB:.2f}" == row["gqa8_gib"]
        assert f"{mla / GiB:.2f}" == row["mla_gib"]
        assert O.sequences_in_budget(budget, mla) == row["mla_seqs"]
    n = 32768
    got = {
        "mha": O.sequences_in_budget(budget, O.kv_cache_bytes(60, 128, 128, n)),
        "gqa8": O.sequences_in_budget(budget, O.kv_cache_bytes(60, 8, 128, n)),
        "mla": O.sequences_in_budget(budget, O.mla_cache_bytes(60, 512, 64, n)),
    }
    assert got == g["seqs_at_32k"]


def test_params_per_layer_printed():
    p = gold("p1_params_macs.json")["params"]
    kw = dict(d_model=p["d_model"], n_heads=p["heads"], head_dim=p["head_dim"])
    mha = O.attention_params_per_layer("mha", **kw)
    gqa = O.attention_params_per_layer("gqa", kv_groups=p["gqa_groups"], **kw)
    mla = O.attention_params_per_layer("mla", d_c=p["d_c"], d_rope=p["d_rope"], **kw)
    assert (mha, gqa, mla) == (p["mha"], p["gqa8"], p["mla"])
    assert f"{mla / mha:.2f}" == p["mla_vs_mha"]
    assert f"{mla / gqa:.2f}" == p["mla_vs_gqa8"]


def test_operation_counts_printed():
    g = gold("p1_params_macs.json")
    m = g["macs"]
    for row in m["rows"]:
        e, a = O.macs_per_head_per_step(row["n"], m["d_model"], m["d_c"], m["head_dim"])
        assert (e, a) == (row["expanded"], row["absorbed"])
        assert f"{e / a:.2f}" == row["saving"]
    r = g["rebuild"]
    assert O.rebuild_absorbed_macs(r["steps"], r["heads"], r["d_model"], r["head_dim"],
                                   r["d_c"]) == r["extra_macs"]


def test_operation_counts_by_brute_force():
    """Count the multiplies of each path on a tiny case by running it."""
    d_model, d_c, d_h, n = 5, 4, 3, 7
    # expanded: keys c@W_uk (n*d_c*d_h), query x@W_q (d_model*d_h), scores K@q (n*d_h)
    # absorbed: x@W_abs (d_model*d_c), scores C@q_lat (n*d_c)
    count = {"e": 0, "a": 0}

    def mm(a_shape, b_shape, key):
        count[key] += a_shape[0] * a_shape[1] * b_shape[1]

    mm((n, d_c), (d_c, d_h), "e")
    mm((1, d_model), (d_model, d_h), "e")
    mm((n, d_h), (d_h, 1), "e")
    mm((1, d_model), (d_model, d_c), "a")
    mm((n, d_c), (d_c, 1), "a")
    assert O.macs_per_head_per_step(n, d_model, d_c, d_h) == (count["e"], count["a"])


# ---------------------------------------------------------------------------
# Softmax and RoPE
# ---------------------------------------------------------------------------


def test_softmax_rows_sum_to_one_and_match_library():
    g = np.random.default_rng(11)
    s = g.normal(0, 5, (64, 37))
    s[:, 5] = -np.inf
    p = O.softmax(s)
    assert np.max(np.abs(p.sum(-1) - 1)) < 1e-12
    assert np.all(p[:, 5] == 0)
    ref = torch.softmax(torch.tensor(s, dtype=torch.float64), dim=-1).numpy()
    assert np.max(np.abs(p - ref)) < 1e-14
    # shift invariance; huge values do not overflow
    assert np.max(np.abs(O.softmax(s + 1e4) - p)) < 1e-12


def _rotation_matrix(pos, d_r, base):
    """Explicit block rotation: plane (i, i + d_r/2) turned by pos*base^(-2i/d_r)."""
    half = d_r // 2
    M = np.zeros((d_r, d_r))
    for i in range(half):
        th = pos * base ** (-2.0 * i / d_r)
        c, s = math.cos(th), math.sin(th)
        M[i, i], M[i, i + half] = c, -s
        M[i + half, i], M[i + half, i + half] = s, c
    return M


def test_rope_matches_explicit_rotation_and_preserves_norm():
    g = np.random.default_rng(12)
    for d_r in (2, 8, 64):
        x = g.normal(size=(5, d_r))
        pos = np.array([0, 1, 17, 4095, 131071])
        y = O.apply_rope(x, pos, 10000.0)
        for k in range(5):
            ref = _rotation_matrix(int(pos[k]), d_r, 10000.0) @ x[k]
            assert np.max(np.abs(y[k] - ref)) < 1e-9
        assert np.max(np.abs(np.linalg.norm(y, axis=-1) - np.linalg.norm(x, axis=-1))) < 1e-12
        assert np.array_equal(O.apply_rope(x[:1], np.array([0]), 10000.0), x[:1])


def test_rope_d2_is_complex_multiplication():
    g = np.random.default_rng(13)
    x = g.normal(size=(9, 2))
    pos = np.arange(9) * 3
    y = O.apply_rope(x, pos, 10000.0)
    z = (x[:, 0] + 1j * x[:, 1]) * np.exp(1j * pos)   # theta_0 = 1 for i = 0
    assert np.max(np.abs(y[:, 0] - z.real)) < 1e-12
    assert np.max(np.abs(y[:, 1] - z.imag)) < 1e-12


def test_rope_relative_position_invariance():
    g = np.random.default_rng(14)
    a, b = g.normal(size=64), g.normal(size=64)
    base = 10000.0
    for m, n in [(0, 5), (100, 105), (131066, 131071), (7, 2), (50007, 50002)]:
        d1 = O.apply_rope(a, m, base) @ O.apply_rope(b, n, base)
        d0 = O.apply_rope(a, 0, base) @ O.apply_rope(b, n - m, base) if n >= m else \
            O.apply_rope(a, m - n, base) @ O.apply_rope(b, 0, base)
        assert abs(d1 - d0) < 1e-9
    # and it does change with the offset
    assert abs(O.apply_rope(a, 0, base) @ O.apply_rope(b, 3, base)
               - O.apply_rope(a, 0, base) @ O.apply_rope(b, 4, base)) > 1e-6


# ---------------------------------------------------------------------------
# Attention: absorbed == materialised == textbook
# ---------------------------------------------------------------------------


def _tiny(seed=0, n_h=4, d_model=32, d_c=16, d_r=8, d_nope=8, d_v=8, L=37):
    g = np.random.default_rng(seed)
    W_dkv = g.normal(0, d_model ** -0.5, (d_model, d_c))
    W_kr = g.normal(0, d_model ** -0.5, (d_model, d_r))
    W_uk = g.normal(0, d_c ** -0.5, (d_c, n_h * d_nope))
    W_uv = g.normal(0, d_c ** -0.5, (d_c, n_h * d_v))
    X = g.normal(size=(L, d_model))
    rows = O.latent_rows(X, W_dkv, W_kr, np.arange(L), 10000.0)
    q = g.normal(size=(1, 2, n_h, d_nope + d_r))
    return dict(W_dkv=W_dkv, W_kr=W_kr, W_uk=W_uk, W_uv=W_uv, X=X, rows=rows, q=q,
                n_h=n_h, d_c=d_c, d_r=d_r, d_nope=d_nope, d_v=d_v, L=L)


def _sdpa_reference(t, n_q, default_scale=False):
    """Textbook attention via torch's scaled_dot_product_attention.

    Keys and values are built explicitly per head: k = [c W_uk_h | k_rope],
    v = c W_uv_h; the query is [q_nope | RoPE(q_rope, pos)].
    """
    d_c, d_nope, d_v, n_h, L = t["d_c"], t["d_nope"], t["d_v"], t["n_h"], t["L"]
    C, KR = t["rows"][:, :d_c], t["rows"][:, d_c:]
    out = np.zeros((n_q, n_h, d_v))
    for h in range(n_h):
        K = np.concatenate([C @ t["W_uk"][:, h * d_nope:(h + 1) * d_nope], KR], axis=1)
        V = C @ t["W_uv"][:, h * d_v:(h + 1) * d_v]
        Q = []
        for i in range(n_q):
            pos = L - n_q + i
            qh = t["q"][0, i, h]
            Q.append(np.concatenate([qh[:d_nope], O.apply_rope(qh[d_nope:], pos, 10000.0)]))
        Q = torch.tensor(np.array(Q))[None, None]
        mask = torch.tensor(np.arange(L)[None, :] <= (L - n_q + np.arange(n_q))[:, None])
        o = torch.nn.functional.scaled_dot_product_attention(
            Q, torch.tensor(K)[None, None], torch.tensor(V)[None, None],
            attn_mask=mask[None, None],
            scale=None if default_scale else O.default_scale(d_nope, t["d_r"]))
        out[:, h] = o[0, 0].numpy()
    return out


def _oracle_out(t, n_q):
    return O.decode_materialised(t["q"][:, :n_q], [t["rows"]], [t["L"]], t["W_uk"], t["W_uv"],
                                 t["d_c"], t["d_nope"], t["d_v"],
                                 O.default_scale(t["d_nope"], t["d_r"]), 10000.0)[0]


@pytest.mark.parametrize("n_q", [1, 2])
def test_materialised_matches_library_attention(n_q):
    t = _tiny(seed=1)
    got = _oracle_out(t, n_q)
    ref = _sdpa_reference(t, n_q)
    assert np.max(np.abs(got - ref)) < 1e-12


def test_absorbed_equals_materialised():
    t = _tiny(seed=2, L=64)
    scale = O.default_scale(t["d_nope"], t["d_r"])
    worst = 0.0
    for h in range(t["n_h"]):
        wuk = O.head_slice(t["W_uk"], h, t["d_nope"])
        wuv = O.head_slice(t["W_uv"], h, t["d_v"])
        for pos in (63, 40):
            a = O.decode_head_absorbed(t["q"][0, 0, h], t["rows"], pos, wuk, wuv, t["d_c"], scale, 1e4)
            m = O.decode_head_materialised(t["q"][0, 0, h], t["rows"], pos, wuk, wuv, t["d_c"], scale, 1e4)
            worst = max(worst, np.max(np.abs(a - m)))
    assert worst <= gold("p1_params_macs.json")["float_noise_bound"]


def test_full_fold_scores_equal_expanded():
    """P1's fold: (x W_q)(c W_uk)^T == (x (W_q W_uk^T)) c^T; and the reversed fold."""
    g = np.random.default_rng(3)
    d_model, d_c, d_h, n = 32, 16, 8, 64
    W_q = g.normal(size=(d_model, d_h))
    W_uk = g.normal(size=(d_c, d_h))
    W_uv = g.normal(size=(d_c, d_h))
    x = g.normal(size=(1, d_model))
    C = g.normal(size=(n, d_c))
    expanded = (x @ W_q) @ (C @ W_uk).T
    W_abs = O.absorb_q_full(W_q, W_uk)
    assert W_abs.shape == (d_model, d_c)
    got = O.scores_absorbed(x, W_abs, C)
    assert np.max(np.abs(got - expanded)) <= 1e-10
    # absorbing the wrong matrix keeps the shape but changes the answer
    wrong = O.scores_absorbed(x, O.absorb_q_full(W_q, W_uv), C)
    assert wrong.shape == got.shape and np.max(np.abs(wrong - expanded)) > 1e-3
    # the transposed order is the same matrix, transposed: harmless
    assert np.max(np.abs((W_uk @ W_q.T).T - W_abs)) == 0.0


def test_rotating_after_absorbing_is_wrong():
    """Rotating the absorbed query does not give the decoupled score."""
    t = _tiny(seed=4, L=16)
    d_c, d_nope, h = t["d_c"], t["d_nope"], 0
    wuk = O.head_slice(t["W_uk"], h, d_nope)
    q = t["q"][0, 0, h]
    C, KR = t["rows"][:, :d_c], t["rows"][:, d_c:]
    correct = C @ (wuk @ q[:d_nope]) + KR @ O.apply_rope(q[d_nope:], 15, 1e4)
    # the broken variant: one rotation applied to the absorbed latent query
    q_lat = wuk @ q[:d_nope]
    broken = C @ O.apply_rope(q_lat, 15, 1e4)
    assert np.max(np.abs(correct - broken)) > 1e-2


def test_full_rank_mla_is_exactly_mha():
    """P1's full-rank check: factor [W_k | W_v] at full rank, run MLA (no RoPE
    block), compare with textbook multi-head attention over X W_k and X W_v."""
    g = np.random.default_rng(5)
    d_model, n_h, d_h, L = 32, 4, 8, 24
    W_k = g.normal(0, 0.4, (d_model, n_h * d_h))
    W_v = g.normal(0, 0.4, (d_model, n_h * d_h))
    W_q = g.normal(0, 0.4, (d_model, n_h * d_h))
    U, S, Vt = np.linalg.svd(np.concatenate([W_k, W_v], axis=1), full_matrices=False)
    d_c = d_model
    W_dkv, W_ukv = U[:, :d_c] * S[:d_c], Vt[:d_c]
    W_uk, W_uv = W_ukv[:, :n_h * d_h], W_ukv[:, n_h * d_h:]
    X = g.normal(size=(L, d_model))
    rows = O.latent_rows(X, W_dkv, np.zeros((d_model, 0)), np.arange(L), 1e4)
    q = (X[-1:] @ W_q).reshape(1, 1, n_h, d_h)
    got = O.decode_materialised(q, [rows], [L], W_uk, W_uv, d_c, d_h, d_h,
                                1 / math.sqrt(d_h), 1e4)[0, 0]
    K = torch.tensor((X @ W_k).reshape(L, n_h, d_h).transpose(1, 0, 2))
    V = torch.tensor((X @ W_v).reshape(L, n_h, d_h).transpose(1, 0, 2))
    Q = torch.tensor(q[0].transpose(1, 0, 2))
    ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V)[:, 0].numpy()
    assert np.max(np.abs(got - ref)) <= gold("p1_params_macs.json")["float_noise_bound"]


def test_single_token_and_identical_rows():
    t = _tiny(seed=6, L=1)
    scale = O.default_scale(t["d_nope"], t["d_r"])
    for h in range(t["n_h"]):
        wuk = O.head_slice(t["W_uk"], h, t["d_nope"])
        wuv = O.head_slice(t["W_uv"], h, t["d_v"])
        o = O.decode_head_materialised(t["q"][0, 0, h], t["rows"], 0, wuk, wuv, t["d_c"], scale, 1e4)
        assert np.max(np.abs(o - t["rows"][0, :t["d_c"]] @ wuv)) < 1e-13
    # identical latent parts with zero rope parts: the scores are all equal,
    # so the output is the mean of the values, which is the one value
    rows = np.repeat(t["rows"][:1], 50, axis=0)
    rows[:, t["d_c"]:] = 0.0
    wuk = O.head_slice(t["W_uk"], 1, t["d_nope"])
    wuv = O.head_slice(t["W_uv"], 1, t["d_v"])
    o = O.decode_head_materialised(t["q"][0, 0, 1], rows, 49, wuk, wuv, t["d_c"], scale, 1e4)
    assert np.max(np.abs(o - rows[0, :t["d_c"]] @ wuv)) < 1e-13


def test_two_queries_are_causal():
    """With n_q = 2 the first query must ignore the newest token entirely."""
    t = _tiny(seed=7, L=20)
    both = _oracle_out(t, 2)
    first_alone = O.decode_materialised(t["q"][:, :1], [t["rows"][:19]], [19], t["W_uk"], t["W_uv"],
                                        t["d_c"], t["d_nope"], t["d_v"],
                                        O.default_scale(t["d_nope"], t["d_r"]), 1e4)[0, 0]
    assert np.max(np.abs(both[0] - first_alone)) < 1e-13
    # perturb the last row: query 0 unchanged, query 1 changes
    t2 = dict(t)
    t2["rows"] = t["rows"].copy()
    t2["rows"][-1] += 1.0
    both2 = _oracle_out(t2, 2)
    assert np.max(np.abs(both2[0] - both[0])) == 0.0
    assert np.max(np.abs(both2[1] - both[1])) > 1e-6


def _latent_queries(t, n_q):
    """q_abs [1, n_q, n_h, d_c + d_r]: per head [W_uk[h]^T q_nope | RoPE(q_rope,
    position)], the absorbed form of the tiny case's queries."""
    d_c, d_nope, n_h, L = t["d_c"], t["d_nope"], t["n_h"], t["L"]
    q_abs = np.zeros((1, n_q, n_h, d_c + t["d_r"]))
    for i in range(n_q):
        for h in range(n_h):
            q = t["q"][0, i, h]
            q_abs[0, i, h, :d_c] = O.head_slice(t["W_uk"], h, d_nope) @ q[:d_nope]
            q_abs[0, i, h, d_c:] = O.apply_rope(q[d_nope:], L - n_q + i, 10000.0)
    return q_abs


@pytest.mark.parametrize("n_q", [1, 2])
def test_latent_core_up_projected_is_library_attention(n_q):
    """The attention core on absorbed queries, up-projected through W_uv[h]
    afterwards, equals torch's scaled_dot_product_attention over the
    explicitly built keys and values (causal for n_q = 2)."""
    t = _tiny(seed=11)
    scale = O.default_scale(t["d_nope"], t["d_r"])
    o_lat = O.decode_latent(_latent_queries(t, n_q), [t["rows"]], [t["L"]], t["d_c"], scale)[0]
    ref = _sdpa_reference(t, n_q)
    for h in range(t["n_h"]):
        got = o_lat[:, h] @ O.head_slice(t["W_uv"], h, t["d_v"])
        assert np.max(np.abs(got - ref[:, h])) < 1e-10


def test_latent_core_closed_forms():
    """One visible key: o_lat is that key's latent row. Equal latent rows and
    zero rope parts: every score is equal and o_lat is the shared row."""
    t = _tiny(seed=12, L=30)
    d_c = t["d_c"]
    q_abs = _latent_queries(t, 1)[0, 0]
    for h in range(t["n_h"]):
        o = O.latent_attention_head(q_abs[h, :d_c], q_abs[h, d_c:], t["rows"], 0, d_c, 0.3)
        assert np.array_equal(o, t["rows"][0, :d_c])
    rows = np.repeat(t["rows"][3:4], 30, axis=0)
    rows[:, d_c:] = 0.0
    o = O.latent_attention_head(q_abs[1, :d_c], q_abs[1, d_c:], rows, 29, d_c, 0.3)
    assert np.max(np.abs(o - rows[0, :d_c])) < 1e-14


ORIG_LATENT_HEAD = O.latent_attention_head


def _latent_mutants():
    def without_position_term(q_lat, q_pe, rows, pos_q, d_c, scale):
        return ORIG_LATENT_HEAD(q_lat, np.zeros_like(q_pe), rows, pos_q, d_c, scale)

    def unscaled(q_lat, q_pe, rows, pos_q, d_c, scale):
        return ORIG_LATENT_HEAD(q_lat, q_pe, rows, pos_q, d_c, 1.0)

    def mask_one_short(q_lat, q_pe, rows, pos_q, d_c, scale):
        return ORIG_LATENT_HEAD(q_lat, q_pe, rows, pos_q - 1, d_c, scale)

    return [without_position_term, unscaled, mask_one_short]


@pytest.mark.parametrize("idx", range(3))
def test_planted_latent_core_mistakes_are_caught(monkeypatch, idx):
    monkeypatch.setattr(O, "latent_attention_head", _latent_mutants()[idx])
    with pytest.raises(AssertionError):
        test_latent_core_up_projected_is_library_attention(2)


def test_default_scale_is_torch_attention_default():
    """The score scale over the full query/key width d_nope + d_r.

    Two anchors outside the oracle: the DeepSeek-V2-shape workload states its
    scale as 1/sqrt(192) (d_nope 128 + d_r 64), and torch's
    scaled_dot_product_attention, called with no scale, divides by the square
    root of the query width, here [q_nope | RoPE(q_rope)]. A scale over
    d_nope alone (P1's toy has no RoPE block, so its 1/sqrt(head_dim) does not
    tell the two apart) fails both.
    """
    assert O.default_scale(128, 64) == 1.0 / math.sqrt(192.0)
    assert O.default_scale(16, 8) == 1.0 / math.sqrt(24.0)
    assert O.default_scale(8, 0) == 1.0 / math.sqrt(8.0)
    for seed, d_nope, d_r in ((21, 8, 8), (22, 16, 4)):
        t = _tiny(seed=seed, d_nope=d_nope, d_r=d_r, L=29)
        got = _oracle_out(t, 2)
        ref = _sdpa_reference(t, 2, default_scale=True)
        assert np.max(np.abs(got - ref)) < 1e-12


def _self_score(x, W_kr, pos):
    """RoPE part of the score of a query whose unrotated rope vector is the
    key's own x W_kr, both at position pos."""
    kr = O.latent_rows(x[None], np.zeros((x.shape[0], 1)), W_kr, np.array([pos]), 1e4)[0, 1:]
    return O.apply_rope(x @ W_kr, pos, 1e4) @ kr


def test_latent_rows_rotate_each_key_by_its_own_position():
    """Pins the position latent_rows rotates each key by.

    [P1 "RoPE, and why the explanations stop here"]: k_rope is computed the
    ordinary way, rotated by its token's position and cached already rotated;
    the query is rotated by its own position at decode time.
      * A key at position 0 is not rotated: its rope block is x W_kr.
      * A query and key at the same position with the same unrotated vector
        score |x W_kr|^2, whatever the position (both rotations cancel).
      * Shifting every key position and the query position by the same
        offset leaves the decode output unchanged (RoPE's relative-position
        property), while shifting the keys alone changes it.
    A key rotated by pos + 1, by -pos, or not at all fails one of these.
    """
    g = np.random.default_rng(23)
    d_model, d_r = 12, 8
    W_kr = g.normal(0, d_model ** -0.5, (d_model, d_r))
    X = g.normal(size=(6, d_model))
    r0 = O.latent_rows(X, np.zeros((d_model, 3)), W_kr, np.zeros(6, dtype=np.int64), 1e4)
    assert np.max(np.abs(r0[:, 3:] - X @ W_kr)) == 0.0
    for pos in (0, 1, 7, 4095, 131071):
        u = X[pos % 6] @ W_kr
        assert abs(_self_score(X[pos % 6], W_kr, pos) - u @ u) < 1e-9 * (1 + u @ u)
    # the whole decode: keys at positions delta .. delta + L - 1, query at the last one
    t = _tiny(seed=24, L=33)
    scale = O.default_scale(t["d_nope"], t["d_r"])
    wuk, wuv = O.head_slice(t["W_uk"], 2, t["d_nope"]), O.head_slice(t["W_uv"], 2, t["d_v"])
    outs = []
    for delta in (0, 5, 1000, 131038):
        rows = O.latent_rows(t["X"], t["W_dkv"], t["W_kr"], np.arange(t["L"]) + delta, 1e4)
        outs.append(O.decode_head_materialised(t["q"][0, 0, 2], rows, t["L"] - 1 + delta,
                                               wuk, wuv, t["d_c"], scale, 1e4))
    for o in outs[1:]:
        assert np.max(np.abs(o - outs[0])) < 1e-12
    rows = O.latent_rows(t["X"], t["W_dkv"], t["W_kr"], np.arange(t["L"]) + 5, 1e4)
    moved = O.decode_head_materialised(t["q"][0, 0, 2], rows, t["L"] - 1, wuk, wuv, t["d_c"],
                                       scale, 1e4)
    assert np.max(np.abs(moved - outs[0])) > 1e-6


# ---------------------------------------------------------------------------
# Paged layout and append
# ---------------------------------------------------------------------------


def test_append_places_rows_by_page_table():
    g = np.random.default_rng(8)
    bs, R, B = 4, 6, 3
    d_model, d_c, d_r = 5, 4, 2
    pt = np.array([[5, 2, -1], [0, 7, 3], [6, 1, 4]], dtype=np.int32)
    cache = g.normal(size=(8, bs, R))
    seq_idx = np.array([0, 1, 1, 2, 0])
    pos = np.array([5, 0, 11, 6, 2])
    x = g.normal(size=(5, d_model))
    W_dkv, W_kr = g.normal(size=(d_model, d_c)), g.normal(size=(d_model, d_r))
    out = O.append_to_paged_cache(cache, x, seq_idx, pos, pt, W_dkv, W_kr, 1e4, bs)
    # brute force: block and slot written out by hand
    where = {0: (2, 1), 1: (0, 0), 2: (3, 3), 3: (1, 2), 4: (5, 2)}
    touched = set()
    for t, (blk, slot) in where.items():
        c = x[t] @ W_dkv
        kr = O.apply_rope(x[t] @ W_kr, pos[t], 1e4)
        assert np.max(np.abs(out[blk, slot] - np.concatenate([c, kr]))) < 1e-12
        touched.add((blk, slot))
    for blk in range(8):
        for slot in range(bs):
            if (blk, slot) not in touched:
                assert np.array_equal(out[blk, slot], cache[blk, slot])
    # gather reads the same rows back in logical order
    seq1 = O.gather_sequence(out, pt, 1, 12, bs)
    assert np.array_equal(seq1[0], out[0, 0]) and np.array_equal(seq1[11], out[3, 3])
    assert np.array_equal(seq1[5], out[7, 1])


# ---------------------------------------------------------------------------
# The pins above must catch plausible mistakes in the oracle
# ---------------------------------------------------------------------------


def _mutants():
    def rope_wrong_sign(x, pos, base):
        x = np.asarray(x, dtype=np.float64)
        half = x.shape[-1] // 2
        if half == 0:
            return x.copy()
        a = O.rope_angles(pos, x.shape[-1], base)
        c, s = np.cos(a), np.sin(a)
        return np.concatenate([x[..., :half] * c + x[..., half:] * s,
                               -x[..., :half] * s + x[..., half:] * c], -1)

    def rope_interleaved(x, pos, base):
        x = np.asarray(x, dtype=np.float64)
        if x.shape[-1] == 0:
            return x.copy()
        a = O.rope_angles(pos, x.shape[-1], base)
        c, s = np.cos(a), np.sin(a)
        y = x.copy()
        y[..., 0::2] = x[..., 0::2] * c - x[..., 1::2] * s
        y[..., 1::2] = x[..., 0::2] * s + x[..., 1::2] * c
        return y

    def no_rope_term(q_head, rows, pos_q, W_uk_h, W_uv_h, d_c, scale, base):
        rows = np.array(rows, dtype=np.float64)
        rows[:, d_c:] = 0.0
        return ORIG_HEAD(q_head, rows, pos_q, W_uk_h, W_uv_h, d_c, scale, base)

    def no_causal(q_head, rows, pos_q, W_uk_h, W_uv_h, d_c, scale, base):
        return ORIG_HEAD(q_head, rows, rows.shape[0] - 1, W_uk_h, W_uv_h, d_c, scale, base)

    def wrong_scale(q_head, rows, pos_q, W_uk_h, W_uv_h, d_c, scale, base):
        return ORIG_HEAD(q_head, rows, pos_q, W_uk_h, W_uv_h, d_c,
                         1 / math.sqrt(W_uk_h.shape[1]), base)

    def swapped_up(q_head, rows, pos_q, W_uk_h, W_uv_h, d_c, scale, base):
        return ORIG_HEAD(q_head, rows, pos_q, W_uv_h, W_uk_h, d_c, scale, base)

    def head_off_by_one(W, h, width):
        W = np.asarray(W, dtype=np.float64)
        n = W.shape[1] // width
        h = (h + 1) % n
        return W[:, h * width:(h + 1) * width]

    def max_without_subtract(s, axis=-1):
        e = np.exp(np.asarray(s, dtype=np.float64) * 1.0001)
        return e / e.sum(axis=axis, keepdims=True)

    return {
        "apply_rope": [rope_wrong_sign, rope_interleaved],
        "decode_head_materialised": [no_rope_term, no_causal, wrong_scale, swapped_up],
        "head_slice": [head_off_by_one],
        "softmax": [max_without_subtract],
    }


ORIG_HEAD = O.decode_head_materialised


@pytest.mark.parametrize("target,idx", [(k, i) for k, v in _mutants().items() for i in range(len(v))])
def test_planted_mistakes_are_caught(monkeypatch, target, idx):
    mutant = _mutants()[target][idx]
    monkeypatch.setattr(O, target, mutant)
    failures = 0
    for check in (lambda: test_materialised_matches_library_attention(2),
                  test_rope_matches_explicit_rotation_and_preserves_norm,
                  test_softmax_rows_sum_to_one_and_match_library):
        try:
            check()
        except AssertionError:
            failures += 1
    assert failures >= 1, f"planted mistake in {target} went unnoticed"


ORIG_LATENT_ROWS = O.latent_rows


def _position_mutants():
    def scale_without_rope_width(d_nope, d_r):
        return 1.0 / math.sqrt(d_nope)

    def scale_over_head_count(d_nope, d_r):
        return 1.0 / (d_nope + d_r)

    def keys_rotated_one_late(x, W_dkv, W_kr, pos, base):
        return ORIG_LATENT_ROWS(x, W_dkv, W_kr, np.asarray(pos) + 1, base)

    def keys_unrotated(x, W_dkv, W_kr, pos, base):
        return ORIG_LATENT_ROWS(x, W_dkv, W_kr, np.zeros_like(np.asarray(pos)), base)

    def keys_rotated_backwards(x, W_dkv, W_kr, pos, base):
        return ORIG_LATENT_ROWS(x, W_dkv, W_kr, -np.asarray(pos), base)

    return {"default_scale": [scale_without_rope_width, scale_over_head_count],
            "latent_rows": [keys_rotated_one_late, keys_unrotated, keys_rotated_backwards]}


@pytest.mark.parametrize("target,idx",
                         [(k, i) for k, v in _position_mutants().items() for i in range(len(v))])
def test_planted_scale_and_position_mistakes_are_caught(monkeypatch, target, idx):
    monkeypatch.setattr(O, target, _position_mutants()[target][idx])
    failures = 0
    for check in (test_default_scale_is_torch_attention_default,
                  test_latent_rows_rotate_each_key_by_its_own_position):
        try:
            check()
        except AssertionError:
            failures += 1
    assert failures >= 1, f"planted mistake in {target} went unnoticed"


# ---------------------------------------------------------------------------
# One layer from the hidden state: x_q in, y = concat_h(o_h) W_o out
# ---------------------------------------------------------------------------


def _layer(seed=7, n_h=3, d_model=24, d_c=16, d_r=4, d_nope=6, d_v=10, lens=(2, 9, 40), n_q=2):
    g = np.random.default_rng(seed)
    W_dkv = g.normal(0, d_model ** -0.5, (d_model, d_c))
    W_kr = g.normal(0, d_model ** -0.5, (d_model, d_r))
    W_q = g.normal(0, d_model ** -0.5, (d_model, n_h * (d_nope + d_r)))
    W_uk = g.normal(0, d_c ** -0.5, (d_c, n_h * d_nope))
    W_uv = g.normal(0, d_c ** -0.5, (d_c, n_h * d_v))
    W_o = g.normal(0, (n_h * d_v) ** -0.5, (n_h * d_v, d_model))
    rows = [O.latent_rows(g.normal(size=(L, d_model)), W_dkv, W_kr, np.arange(L), 1e4)
            for L in lens]
    x_q = g.normal(size=(len(lens), n_q, d_model))
    return dict(W_q=W_q, W_uk=W_uk, W_uv=W_uv, W_o=W_o, rows=rows, lens=np.array(lens),
                x_q=x_q, n_h=n_h, d_c=d_c, d_r=d_r, d_nope=d_nope, d_v=d_v,
                scale=O.default_scale(d_nope, d_r))


def _layer_args(t):
    return (t["x_q"], t["rows"], t["lens"], t["W_q"], t["W_uk"], t["W_uv"], t["W_o"], t["d_c"],
            t["d_nope"], t["d_v"], t["scale"], 1e4)


def test_layer_output_under_permutation_weights():
    """With W_q and W_o permutation matrices, the layer reduces to the
    per-head outputs (pinned above against torch's attention) moved by index:
    q[perm_q[j]] = x_q[j] and y[perm_o[j]] = concat_h(o_h)[j]."""
    t = _layer(seed=8, d_v=10)  # d_model = n_h*(d_nope + d_r) = n_h*d_v = 30
    n_h, dq = t["n_h"], t["d_nope"] + t["d_r"]
    D = n_h * dq
    g = np.random.default_rng(9)
    perm_q, perm_o = g.permutation(D), g.permutation(D)
    assert np.any(perm_q[perm_q] != np.arange(D)) and np.any(perm_o[perm_o] != np.arange(D))
    P_q = np.zeros((D, D))
    P_q[np.arange(D), perm_q] = 1.0
    P_o = np.zeros((D, D))
    P_o[np.arange(D), perm_o] = 1.0
    x_q = g.normal(size=(len(t["lens"]), 2, D))
    q = np.empty_like(x_q)
    q[..., perm_q] = x_q
    o = O.decode_materialised(q.reshape(len(t["lens"]), 2, n_h, dq), t["rows"], t["lens"],
                              t["W_uk"], t["W_uv"], t["d_c"], t["d_nope"], t["d_v"], t["scale"], 1e4)
    want = np.empty((len(t["lens"]), 2, D))
    want[..., perm_o] = o.reshape(len(t["lens"]), 2, D)
    got = O.layer_output_materialised(x_q, t["rows"], t["lens"], P_q, t["W_uk"], t["W_uv"], P_o,
                                      t["d_c"], t["d_nope"], t["d_v"], t["scale"], 1e4)
    assert np.max(np.abs(got - want)) <= 1e-12


def test_layer_output_single_key_closed_form():
    """One cached key gets all the weight, so every head's output is c W_uv[h]
    and the layer output is c W_uv W_o whatever the query."""
    t = _layer(seed=10, lens=(1,), n_q=1)
    c = t["rows"][0][0, :t["d_c"]]
    want = (c @ t["W_uv"]) @ t["W_o"]
    for fn in (O.layer_output_materialised, O.layer_output_absorbed):
        got = fn(*_layer_args(t))[0, 0]
        assert np.max(np.abs(got - want)) <= 1e-12


def test_layer_output_absorbed_equals_materialised():
    """Both folds at once (P1's W_abs = W_q W_uk^T on the query side, P5's
    W_uv W_o on the output side) change nothing but rounding."""
    for seed in (11, 12):
        t = _layer(seed=seed)
        a = O.layer_output_absorbed(*_layer_args(t))
        m = O.layer_output_materialised(*_layer_args(t))
        assert np.all(np.isfinite(m))
        assert np.max(np.abs(a - m)) <= gold("p1_params_macs.json")["float_noise_bound"]
        # the sampled form returns the same rows
        got = O.layer_output_materialised(*_layer_args(t), tokens=[(2, 1), (0, 0)])
        assert np.array_equal(got[(2, 1)], m[2, 1]) and np.array_equal(got[(0, 0)], m[0, 0])


def test_layer_output_absorbing_the_wrong_matrix():
    """P1's "Now break it" row: folding W_uv where W_uk belongs keeps every
    shape and changes the answer."""
    t = _layer(seed=13, d_v=6)  # d_nope == d_v, so the swapped fold has the same shape
    good = O.layer_output_absorbed(*_layer_args(t))
    t2 = dict(t, W_uk=t["W_uv"])
    bad = O.layer_output_absorbed(*_layer_args(t2))
    assert bad.shape == good.shape and np.max(np.abs(bad - good)) > 1e-3


def test_layer_step_under_permutation_output_weights():
    """With W_o a permutation, the step's output is the per-head outputs
    (pinned above) moved by index: y[perm[j]] = concat_h(o_h)[j]."""
    t = _layer(seed=14)
    n_h, d_v = t["n_h"], t["d_v"]
    D = n_h * d_v
    g = np.random.default_rng(15)
    perm = g.permutation(D)
    P = np.zeros((D, D))
    P[np.arange(D), perm] = 1.0
    q = g.normal(size=(len(t["lens"]), 2, n_h, t["d_nope"] + t["d_r"]))
    o = O.decode_materialised(q, t["rows"], t["lens"], t["W_uk"], t["W_uv"], t["d_c"],
                              t["d_nope"], d_v, t["scale"], 1e4)
    want = np.empty((len(t["lens"]), 2, D))
    want[..., perm] = o.reshape(len(t["lens"]), 2, D)
    got = O.layer_step_materialised(q, t["rows"], t["lens"], t["W_uk"], t["W_uv"], P, t["d_c"],
                                    t["d_nope"], d_v, t["scale"], 1e4)
    assert np.max(np.abs(got - want)) <= 1e-12


def test_layer_step_equals_layer_from_hidden_state():
    """Fed q = x_q W_q, the step gives the layer output from x_q."""
    t = _layer(seed=16)
    B, n_q = t["x_q"].shape[:2]
    q = (t["x_q"] @ t["W_q"]).reshape(B, n_q, t["n_h"], t["d_nope"] + t["d_r"])
    a = O.layer_step_materialised(q, t["rows"], t["lens"], t["W_uk"], t["W_uv"], t["W_o"],
                                  t["d_c"], t["d_nope"], t["d_v"], t["scale"], 1e4)
    b = O.layer_output_materialised(*_layer_args(t))
    assert np.max(np.abs(a - b)) <= 1e-12


def _layer_mutants():
    def rope_block_first(W_q, h, d_nope, d_r):
        W_q = np.asarray(W_q, dtype=np.float64)
        dq = d_nope + d_r
        return W_q[:, h * dq + d_r:(h + 1) * dq], W_q[:, h * dq:h * dq + d_r]

    def reversed_latent(W_uv_h, W_o_h):
        return np.asarray(W_uv_h, dtype=np.float64)[::-1] @ np.asarray(W_o_h, dtype=np.float64)

    def no_transpose_fold(W_q_h, W_uk_h):
        return np.asarray(W_q_h, dtype=np.float64) @ np.asarray(W_uk_h, dtype=np.float64)[:, ::-1].T

    return {"head_query_split": [rope_block_first], "fold_value_output": [reversed_latent],
            "absorb_q_full": [no_transpose_fold]}


@pytest.mark.parametrize("target,idx",
                         [(k, i) for k, v in _layer_mutants().items() for i in range(len(v))])
def test_planted_layer_mistakes_are_caught(monkeypatch, target, idx):
    monkeypatch.setattr(O, target, _layer_mutants()[target][idx])
    failures = 0
    for check in (test_layer_output_under_permutation_weights,
                  test_layer_output_single_key_closed_form,
                  test_layer_output_absorbed_equals_materialised):
        try:
            check()
        except AssertionError:
            failures += 1
    assert failures >= 1, f"planted mistake in {target} went unnoticed"


# ---------------------------------------------------------------------------
# fp8 (e4m3) latent cache: the format against torch's float8_e4m3fn
# ---------------------------------------------------------------------------


def _e4m3_values():
    """Every finite e4m3 value, decoded by torch from its byte (254 of 256)."""
    v = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return v[np.isfinite(v)]


def test_e4m3_code_points_are_fixed_points():
    v = _e4m3_values()
    assert len(v) == 254 and v.max() == 448.0 and v.min() == -448.0
    assert np.array_equal(O.e4m3_round(v), v)


def test_e4m3_rounding_matches_torch():
    """Random values, every midpoint between neighbouring codes (the ties),
    their fp32 neighbours, and the subnormal range: the same value as
    torch's float32 -> float8_e4m3fn conversion."""
    g = np.random.default_rng(17)
    pos = np.unique(np.abs(_e4m3_values()))
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    x = np.concatenate([
        g.uniform(-448, 448, 20000).astype(np.float32),
        (g.standard_normal(20000) * 4).astype(np.float32),
        g.uniform(-2.0 ** -5, 2.0 ** -5, 5000).astype(np.float32),
        mids, -mids,
        np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9)),
    ])
    x = x[np.abs(x) <= 448]
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(O.e4m3_round(x.astype(np.float64)), want)


def test_e4m3_saturates_past_448():
    x = np.array([448.0, 450.0, 464.0, 470.0, 1e4, -1e6])
    assert np.array_equal(O.e4m3_round(x), [448, 448, 448, 448, 448, -448])


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
def test_fp8_row_quantiser(dtype):
    g = np.random.default_rng(18)
    rows = g.standard_normal((64, 576))
    rows[3] = 0.0
    codes, scales = O.quantize_rows_fp8(rows, dtype=dtype)
    assert np.array_equal(O.e4m3_round(codes), codes)  # only e4m3 values
    live = np.arange(64) != 3
    assert np.all(np.max(np.abs(codes[live]), axis=1) == 448.0)
    assert scales[3] == 1.0 and np.all(codes[3] == 0)
    assert np.array_equal(scales.astype(dtype).astype(np.float64), scales)
    r = rows.astype(dtype).astype(np.float64)
    deq = O.dequantize_rows_fp8(codes, scales)
    u = np.abs(r) / scales[:, None]  # magnitude in code units
    err = np.abs(deq - r) / scales[:, None]
    tol = np.where(u >= 2.0 ** -6, 2.0 ** -4 * u, 2.0 ** -10) * (1 + 1e-6)
    assert np.all(err <= tol + (1e-6 if dtype == np.float32 else 0))


def test_fp8_cache_error_reaches_the_output():
    """Attention over dequantised rows: the quantisation error passes through
    to the output (P5 "Moving a trained MHA model over"), small but not
    zero."""
    t = _tiny(seed=19, L=200)
    codes, scales = O.quantize_rows_fp8(t["rows"])
    t8 = dict(t, rows=O.dequantize_rows_fp8(codes, scales))
    a, b = _oracle_out(t, 1), _oracle_out(t8, 1)
    rel = np.linalg.norm(a - b) / np.linalg.norm(a)
    assert 1e-4 < rel < 5e-2


def _fp8_mutants():
    def truncating(x):
        x = np.asarray(x, dtype=np.float64)
        a = np.abs(x)
        _, E = np.frexp(a)
        step = np.ldexp(1.0, np.maximum(E - 1, -6) - 3)
        return np.copysign(np.minimum(np.floor(a / step) * step, 448.0), x)

    def no_subnormals(x):
        x = np.asarray(x, dtype=np.float64)
        a = np.abs(x)
        _, E = np.frexp(a)
        step = np.ldexp(1.0, np.maximum(E - 1, -9) - 3)
        return np.copysign(np.minimum(np.rint(a / step) * step, 448.0), x)

    def two_mantissa_bits(x):
        x = np.asarray(x, dtype=np.float64)
        a = np.abs(x)
        _, E = np.frexp(a)
        step = np.ldexp(1.0, np.maximum(E - 1, -6) - 2)
        return np.copysign(np.minimum(np.rint(a / step) * step, 448.0), x)

    return [truncating, no_subnormals, two_mantissa_bits]


@pytest.mark.parametrize("idx", range(3))
def test_planted_fp8_mistakes_are_caught(monkeypatch, idx):
    monkeypatch.setattr(O, "e4m3_round", _fp8_mutants()[idx])
    failures = 0
    for check in (test_e4m3_code_points_are_fixed_points, test_e4m3_rounding_matches_torch):
        try:
            check()
        except AssertionError:
            failures += 1
    assert failures >= 1


def test_prefill_chunk_matches_library_attention():
    """A 24-token chunk at the end of a 40-token sequence (a prefill step):
    each chunk token sees the earlier tokens and itself. Checked against
    torch's attention with the same causal pattern, keys and values built
    per head."""
    g = np.random.default_rng(20)
    n_h, d_model, d_c, d_r, d_nope, d_v, L, n_q = 3, 24, 16, 4, 6, 5, 40, 24
    W_dkv = g.normal(0, d_model ** -0.5, (d_model, d_c))
    W_kr = g.normal(0, d_model ** -0.5, (d_model, d_r))
    W_uk = g.normal(0, d_c ** -0.5, (d_c, n_h * d_nope))
    W_uv = g.normal(0, d_c ** -0.5, (d_c, n_h * d_v))
    rows = O.latent_rows(g.normal(size=(L, d_model)), W_dkv, W_kr, np.arange(L), 1e4)
    q = g.normal(size=(1, n_q, n_h, d_nope + d_r))
    scale = O.default_scale(d_nope, d_r)
    got = O.decode_materialised(q, [rows], [L], W_uk, W_uv, d_c, d_nope, d_v, scale, 1e4)[0]
    C, KR = rows[:, :d_c], rows[:, d_c:]
    pos = L - n_q + np.arange(n_q)
    mask = torch.tensor(np.arange(L)[None, :] <= pos[:, None])
    for h in range(n_h):
        K = np.concatenate([C @ W_uk[:, h * d_nope:(h + 1) * d_nope], KR], axis=1)
        V = C @ W_uv[:, h * d_v:(h + 1) * d_v]
        Q = np.stack([np.concatenate([q[0, i, h, :d_nope],
                                      O.apply_rope(q[0, i, h, d_nope:], pos[i], 1e4)])
                      for i in range(n_q)])
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.tensor(Q)[None], torch.tensor(K)[None], torch.tensor(V)[None],
            attn_mask=mask[None], scale=scale)[0].numpy()
        assert np.max(np.abs(got[:, h] - ref)) < 1e-12
