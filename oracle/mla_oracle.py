"""fp64 CPU oracle for Multi-head Latent Attention decode over a latent KV cache.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it. The
CUDA library never calls it, and it shares no code with the CUDA path.

It computes attention the slow, explicit way: per head it materialises
k = c·W_uk and v = c·W_uv for every cached token and then runs textbook softmax
attention. The absorbed form is here too, but only so the tests can check the
algebra.

Sources. Each function names the page and section it follows:
  [P1] "Multi-head Latent Attention: the KV cache, compressed" (paperfordummies.in)
  [P2] "Multi-Head Latent Attention (MLA)" (superteams.ai glossary)
  [P4] "DeepSeek V3 Multi-Head Latent Attention (MLA): How It Slashes KV Cache Memory"
  [P5] "Multi-head Latent Attention and KV Cache Compression" (jongkwan.dev)

Readings taken where the pages leave a step open:
  * RoPE pairs dimension i with dimension i + d_r/2 (the "half-split" form),
    with angle pos * base^(-2i/d_r). P1 calls ``apply_rope`` but does not
    print it.
  * A token's position is its 0-based index in its sequence. ``seq_len``
    already counts the n_q new tokens, so query i sits at L - n_q + i and
    sees keys j <= L - n_q + i.
  * Each head has its own q = [q_nope | q_rope]. One k_rope is shared by all
    heads [P1 "RoPE, and why the explanations stop here"; P2 "The Mechanism"].
  * The score scale is 1/sqrt(d_nope + d_r).
  * The paged layout: token j of sequence b is stored in row
    ``page_table[b][j // block_size] * block_size + j % block_size``.

Parity status: every function here is pinned by a ``-m "not gpu"`` test in
``tests/test_oracle_pins.py``. The pins are closed forms, printed values,
textbook routines, invariants and brute-force checks. The exceptions are P1's
printed score vectors: the script that drew those inputs is not on the pages,
so those vectors are "parity unpinned" and the oracle does not try to match
them.
"""
from __future__ import annotations

import math

import numpy as np

# ---------------------------------------------------------------------------
# Cache and parameter arithmetic
# ---------------------------------------------------------------------------


def kv_cache_bytes(layers, kv_heads, head_dim, seq_len, dtype_bytes=2, batch=1):
    """Cache bytes of a standard multi-head (or grouped-query) KV cache.

    [P1] "The one formula" (the MHA line) and "The code" (``kv_cache_bytes``).
    K and V are both stored, hence the leading 2. Grouped-query attention is
    this same formula with kv_heads set to the group count.
    """
    return 2 * layers * kv_heads * head_dim * seq_len * dtype_bytes * batch


def mla_cache_bytes(layers, d_c, d_rope, seq_len, dtype_bytes=2, batch=1):
    """Cache bytes of an MLA latent cache.

    [P1] "The one formula" (the MLA line) and "The code" (``mla_cache_bytes``);
    [P2] "The Mechanism". Each token stores one [c | k_rope] row per layer,
    shared by every head.
    """
    return layers * (d_c + d_rope) * seq_len * dtype_bytes * batch


def sequences_in_budget(budget_bytes, bytes_per_sequence):
    """Whole sequences that fit in a cache budget.

    [P1] "Where the saving actually lands": the count of concurrent sequences
    that fit on one card.
    """
    return int(budget_bytes // bytes_per_sequence)


def attention_params_per_layer(kind, d_model, n_heads, head_dim, kv_groups=None,
                               d_c=None, d_rope=None):
    """Weight count of one attention layer.

    [P1] "What it costs, said plainly". The MLA count is the sum of W_q
    (d_model -> n_h*(head_dim + d_rope)), W_dkv (d_model -> d_c), W_kr
    (d_model -> d_rope), W_uk and W_uv (d_c -> n_h*head_dim each) and W_o
    (n_h*head_dim -> d_model). There is no query compression [P1 same
    section]. That weight inventory reproduces the page's printed total
    exactly. The pin test checks this.
    """
    d_all = n_heads * head_dim
    if kind == "mha":
        return 4 * d_model * d_all
    if kind == "gqa":
        kv = kv_groups * head_dim
        return d_model * d_all + 2 * d_model * kv + d_all * d_model
    if kind == "mla":
        w_q = d_model * n_heads * (head_dim + d_rope)
        w_dkv = d_model * d_c
        w_kr = d_model * d_rope
        w_uk = d_c * d_all
        w_uv = d_c * d_all
        w_o = d_all * d_model
        return w_q + w_dkv + w_kr + w_uk + w_uv + w_o
    raise ValueError(kind)


def macs_per_head_per_step(n_cached, d_model, d_c, head_dim):
    """Multiply-accumulates per head per decode step, expanded vs absorbed.

    [P1] "Absorption: the part that makes it free" (the operation-count table).
    Expanded: re-expand each cached latent into a key (n*d_c*d_h), project the
    query (d_model*d_h), then score (n*d_h). Absorbed: project the query
    straight into latent space (d_model*d_c), then score against the latent
    (n*d_c).
    Returns (expanded, absorbed).
    """
    expanded = n_cached * d_c * head_dim + d_model * head_dim + n_cached * head_dim
    absorbed = d_model * d_c + n_cached * d_c
    return expanded, absorbed


def rebuild_absorbed_macs(steps, n_heads, d_model, head_dim, d_c):
    """MACs wasted by rebuilding W_abs = W_q W_uk^T on every decode step.

    [P1] "Now break it" (the row about rebuilding the absorbed matrix inside
    the decode loop). Each step redoes one (d_model x d_h) @ (d_h x d_c)
    product per head.
    """
    return steps * n_heads * d_model * head_dim * d_c


# ---------------------------------------------------------------------------
# Building blocks of the method
# ---------------------------------------------------------------------------


def softmax(s, axis=-1):
    """Numerically stable softmax: subtract the max, exponentiate, normalise.

    P1 calls it in "The code" (``attention_via_latent``) but does not print
    it; this is the textbook definition. Entries equal to -inf get weight 0.
    """
    s = np.asarray(s, dtype=np.float64)
    m = np.max(s, axis=axis, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=axis, keepdims=True)


def rope_angles(pos, d_r, base):
    """Rotation angles pos * base^(-2i/d_r) for i < d_r/2, in fp64.

    [P1] "RoPE, and why the explanations stop here": RoPE turns q and k by an
    angle that grows with their position. The frequency ladder is the
    standard rotary one, with base 10000 for every workload here.
    """
    assert d_r % 2 == 0
    half = d_r // 2
    inv_freq = np.power(float(base), -2.0 * np.arange(half, dtype=np.float64) / d_r)
    return np.asarray(pos, dtype=np.float64)[..., None] * inv_freq


def apply_rope(x, pos, base):
    """Rotate the last axis of x (width d_r) by position ``pos``.

    Reading (P1 does not print ``apply_rope``): pair dimension i with
    i + d_r/2 and rotate each pair by the angle from :func:`rope_angles`.
    ``pos`` broadcasts against x's leading axes.
    """
    x = np.asarray(x, dtype=np.float64)
    d_r = x.shape[-1]
    if d_r == 0:
        return x.copy()
    half = d_r // 2
    ang = rope_angles(pos, d_r, base)
    cos, sin = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * cos - x2 * sin, x1 * sin + x2 * cos], axis=-1)


def latent_rows(x, W_dkv, W_kr, pos, base):
    """One cache row per token: [c = x W_dkv | k_rope = RoPE(x W_kr, pos)].

    [P1] "The code" (``latent``) and "RoPE, and why the explanations stop
    here" (the decoupled block is computed the ordinary way and cached
    already rotated); [P4] "Low-Rank Key-Value Joint Compression";
    [P5] "Caching one latent vector".
    x: [T, d_model]; W_dkv: [d_model, d_c]; W_kr: [d_model, d_r]; pos: [T].
    Returns [T, d_c + d_r] in fp64.
    """
    x = np.asarray(x, dtype=np.float64)
    c = x @ np.asarray(W_dkv, dtype=np.float64)
    kr = apply_rope(x @ np.asarray(W_kr, dtype=np.float64), pos, base)
    return np.concatenate([c, kr], axis=-1)


def paged_row_index(page_table, b, j, block_size):
    """Physical cache row that holds token j of sequence b.

    The pages say nothing about paging. The reading taken here is that block
    ``page_table[b][j // block_size]`` holds tokens in order, one row each.
    """
    return int(page_table[b][j // block_size]) * block_size + j % block_size


def append_to_paged_cache(cache, x, seq_idx, pos, page_table, W_dkv, W_kr, base,
                          block_size):
    """Compute each new token's row and write it into a copy of the paged cache.

    cache: [num_blocks, block_size, R]. Returns the updated copy in fp64.
    Rows that no token writes keep their old contents.
    """
    out = np.array(cache, dtype=np.float64, copy=True)
    R = out.shape[-1]
    flat = out.reshape(-1, R)
    rows = latent_rows(x, W_dkv, W_kr, pos, base)
    for t in range(rows.shape[0]):
        r = paged_row_index(page_table, int(seq_idx[t]), int(pos[t]), block_size)
        flat[r] = rows[t]
    return out


def gather_sequence(cache, page_table, b, L, block_size):
    """Logical rows [L, R] of sequence b, read out of the paged cache."""
    R = cache.shape[-1]
    flat = np.asarray(cache).reshape(-1, R)
    idx = [paged_row_index(page_table, b, j, block_size) for j in range(L)]
    return np.asarray(flat[idx], dtype=np.float64)


# ---------------------------------------------------------------------------
# Decode attention, materialised (the oracle proper)
# ---------------------------------------------------------------------------


def head_slice(W, h, width):
    """Columns of head h in a [rows, n_h*width] matrix (P1's convention)."""
    return np.asarray(W, dtype=np.float64)[:, h * width:(h + 1) * width]


def decode_head_materialised(q_head, rows, pos_q, W_uk_h, W_uv_h, d_c, scale, base):
    """Attention output of one head for one query token, keys materialised.

    [P1] "The code" (``attention_via_latent``: re-expand K and V from the
    latent, then textbook attention) and "RoPE, and why the explanations stop
    here" (score = content part + decoupled RoPE part); [P4] "Low-Rank
    Key-Value Joint Compression" (k = W_UK c, v = W_UV c); [P5] "The
    absorption trick and decoupled RoPE" (the final score is the sum of the
    two inner products).

    q_head: [d_nope + d_r], RoPE not yet applied. rows: [L, d_c + d_r] logical
    cache rows. Keys j > pos_q are masked out (causal). W_uk_h: [d_c, d_nope];
    W_uv_h: [d_c, d_v].
    """
    q_head = np.asarray(q_head, dtype=np.float64)
    rows = np.asarray(rows, dtype=np.float64)
    d_nope = W_uk_h.shape[1]
    C = rows[:, :d_c]
    KR = rows[:, d_c:]
    q_nope = q_head[:d_nope]
    q_rope = apply_rope(q_head[d_nope:], pos_q, base)
    K = C @ W_uk_h                       # [L, d_nope]  materialised keys
    V = C @ W_uv_h                       # [L, d_v]     materialised values
    s = (K @ q_nope + KR @ q_rope) * scale
    L = rows.shape[0]
    s = np.where(np.arange(L) <= pos_q, s, -np.inf)
    p = softmax(s)
    return p @ V


def decode_materialised(q, seq_rows, seq_lens, W_uk, W_uv, d_c, d_nope, d_v,
                        scale, base, samples=None):
    """Decode outputs for a batch. This is the oracle the CUDA path is checked against.

    q: [B, n_q, n_h, d_nope + d_r]. seq_rows: a list whose entry b holds the
    logical rows [L_b, R] of sequence b (entries that no sample needs may be
    None). ``samples`` is None for every (b, i, h), or an iterable of (b, i, h)
    triples. Returns the [B, n_q, n_h, d_v] array (entries that were not
    sampled stay NaN) when samples is None, else a dict keyed by (b, i, h).
    """
    q = np.asarray(q, dtype=np.float64)
    B, n_q, n_h, _ = q.shape
    want = samples
    if want is None:
        want = [(b, i, h) for b in range(B) for i in range(n_q) for h in range(n_h)]
    res = {}
    wuk = [None] * n_h
    wuv = [None] * n_h
    for (b, i, h) in want:
        if wuk[h] is None:
            wuk[h] = head_slice(W_uk, h, d_nope)
            wuv[h] = head_slice(W_uv, h, d_v)
        L = int(seq_lens[b])
        pos_q = L - n_q + i
        res[(b, i, h)] = decode_head_materialised(
            q[b, i, h], seq_rows[b][:L], pos_q, wuk[h], wuv[h], d_c, scale, base)
    if samples is not None:
        return res
    out = np.full((B, n_q, n_h, d_v), np.nan)
    for (b, i, h), v in res.items():
        out[b, i, h] = v
    return out


# ---------------------------------------------------------------------------
# Absorbed forms (used only to pin the algebra; the GPU path is checked
# against the materialised form above)
# ---------------------------------------------------------------------------


def absorb_q_full(W_q_h, W_uk_h):
    """W_abs = W_q_h W_uk_h^T, shape (d_model, d_c), built once at load.

    [P1] "Store the archive, not the files" and "Absorption: the part that
    makes it free" (``absorb_q_into_latent``).
    """
    return np.asarray(W_q_h, dtype=np.float64) @ np.asarray(W_uk_h, dtype=np.float64).T


def scores_absorbed(x, W_abs, C):
    """(x W_abs) C^T: scores against the latent, keys never built.

    [P1] "The code" (``scores_absorbed``).
    """
    return (np.asarray(x, dtype=np.float64) @ W_abs) @ np.asarray(C, dtype=np.float64).T


def decode_head_absorbed(q_head, rows, pos_q, W_uk_h, W_uv_h, d_c, scale, base):
    """The same head output as :func:`decode_head_materialised`, computed absorbed.

    q_lat = W_uk_h q_nope goes into latent space [P5 "The absorption trick and
    decoupled RoPE", first identity]. The latent output o_lat = sum_j p_j c_j
    is up-projected through W_uv at the end [P5 same section, value side].
    """
    q_head = np.asarray(q_head, dtype=np.float64)
    rows = np.asarray(rows, dtype=np.float64)
    d_nope = W_uk_h.shape[1]
    C, KR = rows[:, :d_c], rows[:, d_c:]
    q_lat = W_uk_h @ q_head[:d_nope]
    q_pe = apply_rope(q_head[d_nope:], pos_q, base)
    s = (C @ q_lat + KR @ q_pe) * scale
    s = np.where(np.arange(rows.shape[0]) <= pos_q, s, -np.inf)
    p = softmax(s)
    o_lat = p @ C
    return o_lat @ W_uv_h


def latent_attention_head(q_lat, q_pe, rows, pos_q, d_c, scale):
    """The latent output of one head for one query, before the value
    up-projection: o_lat = sum_j p_j c_j with p = softmax over the visible
    keys (j <= pos_q) of scale * (q_lat . c_j + q_pe . k_rope_j).

    [P5] "The absorption trick and decoupled RoPE" (the content score is
    q_lat . c with q_lat = W_uk^T q_nope, the position score q_pe . k_rope
    is added, and the output side keeps the weighted latent sum, W_uv being
    applied once afterwards); [P1] "RoPE, and why the explanations stop
    here" (the position part is its own inner product). q_pe is already
    rotated; rows: [L, d_c + d_r] logical cache rows.
    """
    q_lat = np.asarray(q_lat, dtype=np.float64)
    q_pe = np.asarray(q_pe, dtype=np.float64)
    rows = np.asarray(rows, dtype=np.float64)
    C, KR = rows[:, :d_c], rows[:, d_c:]
    s = (C @ q_lat + KR @ q_pe) * scale
    s = np.where(np.arange(rows.shape[0]) <= pos_q, s, -np.inf)
    return softmax(s) @ C


def decode_latent(q_abs, seq_rows, seq_lens, d_c, scale, samples=None):
    """latent_attention_head over a batch: q_abs [B, n_q, n_h, d_c + d_r]
    holds per head [q_lat | q_pe]; query i of sequence b sits at position
    seq_lens[b] - n_q + i. Returns [B, n_q, n_h, d_c] (NaN where not
    sampled) when samples is None, else a dict keyed by (b, i, h)."""
    q_abs = np.asarray(q_abs, dtype=np.float64)
    B, n_q, n_h, _ = q_abs.shape
    want = samples
    if want is None:
        want = [(b, i, h) for b in range(B) for i in range(n_q) for h in range(n_h)]
    res = {}
    for (b, i, h) in want:
        L = int(seq_lens[b])
        res[(b, i, h)] = latent_attention_head(q_abs[b, i, h, :d_c], q_abs[b, i, h, d_c:],
                                               seq_rows[b][:L], L - n_q + i, d_c, scale)
    if samples is not None:
        return res
    out = np.full((B, n_q, n_h, d_c), np.nan)
    for (b, i, h), v in res.items():
        out[b, i, h] = v
    return out


def default_scale(d_nope, d_r):
    """Score scale 1/sqrt(d_nope + d_r). A head's query/key width is d_nope + d_r."""
    return 1.0 / math.sqrt(d_nope + d_r)


# ---------------------------------------------------------------------------
# One attention layer from the hidden state: x_q in, y out
# ---------------------------------------------------------------------------


def head_query_split(W_q, h, d_nope, d_r):
    """(W_q,nope[h], W_qr[h]) of head h from W_q [d_model, n_h*(d_nope + d_r)].

    Each head's query block is [q_nope | q_rope]; W_qr[h] is the matrix P1
    calls ``W_qr`` in "The code" (``decoupled_score``).
    """
    W_q = np.asarray(W_q, dtype=np.float64)
    dq = d_nope + d_r
    return W_q[:, h * dq:h * dq + d_nope], W_q[:, h * dq + d_nope:(h + 1) * dq]


def layer_output_materialised(x_q, seq_rows, seq_lens, W_q, W_uk, W_uv, W_o, d_c, d_nope,
                              d_v, scale, base, tokens=None):
    """Layer output y = concat_h(o_h) W_o, with every key and value materialised.

    q = x_q W_q per head [P1 "The code", ``attention_via_latent``: the query
    is the hidden state times W_q, cut into heads]; o_h is
    :func:`decode_head_materialised`; the heads are concatenated and
    projected by W_o [n_h*d_v, d_model] (reading: the pages list W_o among the
    layer's weights, P1 "What it costs, said plainly", but print no output
    projection; this is the usual one). Nothing is rounded: q is never
    stored in this form.

    x_q: [B, n_q, d_model]. ``tokens`` is None for every (b, i), or an
    iterable of (b, i) pairs. Returns [B, n_q, d_model] (rows not computed
    stay NaN) when tokens is None, else a dict keyed by (b, i).
    """
    x_q = np.asarray(x_q, dtype=np.float64)
    B, n_q, _ = x_q.shape
    W_q = np.asarray(W_q, dtype=np.float64)
    W_o = np.asarray(W_o, dtype=np.float64)
    n_h = W_o.shape[0] // d_v
    d_r = W_q.shape[1] // n_h - d_nope
    want = tokens if tokens is not None else [(b, i) for b in range(B) for i in range(n_q)]
    res = {}
    for (b, i) in want:
        q = (x_q[b, i] @ W_q).reshape(n_h, d_nope + d_r)
        L = int(seq_lens[b])
        pos_q = L - n_q + i
        o = np.concatenate([
            decode_head_materialised(q[h], seq_rows[b][:L], pos_q, head_slice(W_uk, h, d_nope),
                                     head_slice(W_uv, h, d_v), d_c, scale, base)
            for h in range(n_h)])
        res[(b, i)] = o @ W_o
    if tokens is not None:
        return res
    out = np.full((B, n_q, W_o.shape[1]), np.nan)
    for (b, i), v in res.items():
        out[b, i] = v
    return out


def fold_value_output(W_uv_h, W_o_h):
    """W_vo[h] = W_uv[h] W_o[h], shape (d_c, d_model), built once at load.

    [P5] "The absorption trick and decoupled RoPE": the value-side
    up-projection folds into the output projection the way W_uk folds into
    the query side. W_o_h is the d_v rows of W_o that head h's output meets.
    """
    return np.asarray(W_uv_h, dtype=np.float64) @ np.asarray(W_o_h, dtype=np.float64)


def layer_output_absorbed(x_q, seq_rows, seq_lens, W_q, W_uk, W_uv, W_o, d_c, d_nope, d_v,
                          scale, base, tokens=None):
    """:func:`layer_output_materialised` with both folds done first.

    Per head: W_abs[h] = W_q,nope[h] W_uk[h]^T [P1 "Store the archive, not the
    files" and "The code", ``absorb_q_into_latent``], W_vo[h] =
    :func:`fold_value_output`. Then for each query token, content scores
    (x_q W_abs[h]) c_j^T plus the decoupled part RoPE(x_q W_qr[h]) k_rope_j^T
    [P1 "The code", ``decoupled_score``], softmax, o_lat = sum_j p_j c_j, and
    y = sum_h o_lat[h] W_vo[h]. Used only to pin the algebra.
    """
    x_q = np.asarray(x_q, dtype=np.float64)
    B, n_q, d_model = x_q.shape
    W_o = np.asarray(W_o, dtype=np.float64)
    n_h = W_o.shape[0] // d_v
    d_r = np.asarray(W_q).shape[1] // n_h - d_nope
    W_abs, W_qr, W_vo = [], [], []
    for h in range(n_h):
        wqn, wqr = head_query_split(W_q, h, d_nope, d_r)
        W_abs.append(absorb_q_full(wqn, head_slice(W_uk, h, d_nope)))
        W_qr.append(wqr)
        W_vo.append(fold_value_output(head_slice(W_uv, h, d_v), W_o[h * d_v:(h + 1) * d_v]))
    want = tokens if tokens is not None else [(b, i) for b in range(B) for i in range(n_q)]
    res = {}
    for (b, i) in want:
        L = int(seq_lens[b])
        pos_q = L - n_q + i
        rows = np.asarray(seq_rows[b][:L], dtype=np.float64)
        C, KR = rows[:, :d_c], rows[:, d_c:]
        y = np.zeros(d_model)
        for h in range(n_h):
            s = (C @ (x_q[b, i] @ W_abs[h]) + KR @ apply_rope(x_q[b, i] @ W_qr[h], pos_q, base))
            s = np.where(np.arange(L) <= pos_q, s * scale, -np.inf)
            y += (softmax(s) @ C) @ W_vo[h]
        res[(b, i)] = y
    if tokens is not None:
        return res
    out = np.full((B, n_q, d_model), np.nan)
    for (b, i), v in res.items():
        out[b, i] = v
    return out


def layer_step_materialised(q, seq_rows, seq_lens, W_uk, W_uv, W_o, d_c, d_nope, d_v, scale,
                            base):
    """One layer's decode step from the projected queries: every head's
    materialised attention (:func:`decode_materialised`), the heads
    concatenated, then the output projection y = concat_h(o_h) W_o.

    q: [B, n_q, n_h, d_nope + d_r] before RoPE. W_o: [n_h*d_v, d_model] (the
    reading of :func:`layer_output_materialised`). Returns y [B, n_q, d_model].
    The query projection stays with the caller, as for the decode step.
    """
    o = decode_materialised(q, seq_rows, seq_lens, W_uk, W_uv, d_c, d_nope, d_v, scale, base)
    B, n_q, n_h, _ = o.shape
    return o.reshape(B, n_q, n_h * d_v) @ np.asarray(W_o, dtype=np.float64)


# ---------------------------------------------------------------------------
# fp8 (e4m3) latent cache with one scale per row
# ---------------------------------------------------------------------------

E4M3_MAX = 448.0  # 1.75 * 2^8, the largest finite e4m3 value


def e4m3_round(x):
    """Nearest e4m3 value of each element (ties to even), in fp64.

    The e4m3 format ("fn" variant): 1 sign bit, 4 exponent bits with bias 7,
    3 mantissa bits; below 2^-6 the values are subnormal, in steps of 2^-9;
    the largest finite value is 448 and there are no infinities. A magnitude
    above 448 saturates to 448 (reading: the row quantiser scales every row
    so that none does).

    The pages quantise the latent vector only in passing [P5 "Moving a
    trained MHA model over": quantisation on top of the latent cache, and its
    error passing through the up-projection]; they fix neither the format
    nor the scale granularity.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, E = np.frexp(a)                    # a = m * 2^E with m in [0.5, 1)
    e = np.maximum(E - 1, -6)             # binade exponent; subnormals share 2^-6's step
    step = np.ldexp(1.0, e - 3)           # 3 mantissa bits
    q = np.minimum(np.rint(a / step) * step, E4M3_MAX)  # rint: ties to even
    return np.copysign(q, x)


def quantize_rows_fp8(rows, dtype=np.float64):
    """One cache row -> (e4m3 values, one scale), row by row.

    scale = max|row| / 448 and code = e4m3_round(row / scale), so each row's
    largest element becomes +-448 exactly. A row of zeros gets scale 1.
    ``dtype`` is the precision the scale and the division are computed in
    (np.float32 mirrors a kernel that quantises fp32 accumulators).
    Returns (codes [..., R] fp64 holding e4m3 values, scales [...] fp64).
    """
    r = np.asarray(rows, dtype=dtype)
    amax = np.max(np.abs(r), axis=-1)
    scale = np.where(amax > 0, amax / dtype(E4M3_MAX), dtype(1.0)).astype(dtype)
    codes = e4m3_round((r / scale[..., None]).astype(dtype))
    return codes, scale.astype(np.float64)


def dequantize_rows_fp8(codes, scales):
    """Cache rows back from e4m3 values and their row scales: code * scale."""
    return np.asarray(codes, dtype=np.float64) * np.asarray(scales, dtype=np.float64)[..., None]
