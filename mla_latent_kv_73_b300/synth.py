"""Seeded synthetic inputs for the MLA decode workloads.

This module only draws random numbers, rounds them to the workload's dtype and
builds page tables. It holds none of the method's arithmetic. The tests, the
benchmark and the oracle-side checks all get their inputs from here, so the
CUDA path and the fp64 oracle see exactly the same values.

Every array comes from ``numpy.random.default_rng([seed, stream, ...])``, so one
sequence's cache rows can be regenerated without drawing the others.

Distributions:
  * Weights are N(0, 1/fan_in), where fan_in is the input width: d_model for
    W_dkv, W_kr and W_q; d_c for W_uk and W_uv; n_h*d_v for W_o.
  * Hidden states are N(0, 1).
  * Cache rows [c | k_rope] and queries [q_nope | q_rope] are drawn directly
    as N(0, 1). That is the distribution x·W_dkv and x·W_q have when
    x ~ N(0, 1) and the weights are N(0, 1/d_model).
  * In bf16 workloads every value is rounded to the nearest bf16 (ties to
    even) on the host, so both sides start from identical numbers.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

# Sub-stream ids
_S_WEIGHTS, _S_LENS, _S_PAGES, _S_CACHE, _S_Q, _S_X, _S_FP8, _S_QLAT = 1, 2, 3, 4, 5, 6, 7, 8


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    n_h: int
    d_model: int
    d_c: int
    d_r: int
    d_nope: int
    d_v: int
    batch: int
    n_q: int
    len_lo: int          # seq_lens drawn uniform in [len_lo, len_hi] (inclusive)
    len_hi: int
    dtype: str           # "f32" or "bf16"
    seed: int
    block_size: int = 64
    rope_base: float = 10000.0

    @property
    def R(self):
        return self.d_c + self.d_r

    @property
    def scale(self):
        return 1.0 / math.sqrt(self.d_nope + self.d_r)

    @property
    def elem_bytes(self):
        return 4 if self.dtype == "f32" else 2


WORKLOADS = {
    # 1 layer, fp32, batch 2, 128 cached tokens, 1 query token.
    "tiny_fp32": Workload("tiny_fp32", n_h=4, d_model=64, d_c=32, d_r=8, d_nope=16,
                          d_v=16, batch=2, n_q=1, len_lo=128, len_hi=128,
                          dtype="f32", seed=0),
    # DeepSeek-V2 shape, batch 16, every sequence 4096 tokens.
    "dsv2_b16_l4096": Workload("dsv2_b16_l4096", n_h=128, d_model=5120, d_c=512,
                               d_r=64, d_nope=128, d_v=128, batch=16, n_q=1,
                               len_lo=4096, len_hi=4096, dtype="bf16", seed=1),
    # DeepSeek-V2 shape, batch 64, lengths uniform in [512, 32768].
    "dsv2_b64_ragged": Workload("dsv2_b64_ragged", n_h=128, d_model=5120, d_c=512,
                                d_r=64, d_nope=128, d_v=128, batch=64, n_q=1,
                                len_lo=512, len_hi=32768, dtype="bf16", seed=2),
    # DeepSeek-V2 shape, batch 4, 131072 tokens each (2 of them new queries).
    "dsv2_b4_l131072_nq2": Workload("dsv2_b4_l131072_nq2", n_h=128, d_model=5120,
                                    d_c=512, d_r=64, d_nope=128, d_v=128, batch=4,
                                    n_q=2, len_lo=131072, len_hi=131072,
                                    dtype="bf16", seed=3),
    # 16 heads, d_model 2048, batch 256, lengths uniform in [1024, 8192].
    "nh16_b256_ragged": Workload("nh16_b256_ragged", n_h=16, d_model=2048, d_c=512,
                                 d_r=64, d_nope=128, d_v=128, batch=256, n_q=1,
                                 len_lo=1024, len_hi=8192, dtype="bf16", seed=4),
}

# A prefill step (not one of the decode workloads): 512 new tokens per
# sequence appended and attended in one call, at the end of 4096-token
# sequences (the count includes the new tokens), DeepSeek-V2 shape.
WORKLOADS["dsv2_prefill_b4_c512_l4096"] = Workload(
    "dsv2_prefill_b4_c512_l4096", n_h=128, d_model=5120, d_c=512, d_r=64, d_nope=128, d_v=128,
    batch=4, n_q=512, len_lo=4096, len_hi=4096, dtype="bf16", seed=5)

WORKLOAD_ORDER = ["tiny_fp32", "dsv2_b16_l4096", "dsv2_b64_ragged",
                  "dsv2_b4_l131072_nq2", "nh16_b256_ragged"]


def rng(seed, *stream):
    return np.random.default_rng([int(seed), *[int(s) for s in stream]])


def round_bf16(a):
    """Round float32 values to the nearest bf16 (ties to even).

    Returns (values as float32, raw bf16 bits as uint16). Inputs must be
    finite.
    """
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    bits = u.astype(np.uint16)
    vals = (bits.astype(np.uint32) << 16).view(np.float32)
    return vals, bits


def to_dtype(a, dtype):
    """float32 array -> (values exactly representable in dtype, storage array)."""
    if dtype == "f32":
        v = np.ascontiguousarray(a, dtype=np.float32)
        return v, v
    return round_bf16(a)


def normal(g, shape, std=1.0):
    return (g.standard_normal(size=shape, dtype=np.float32) * np.float32(std))


@dataclasses.dataclass
class Weights:
    W_dkv: np.ndarray   # [d_model, d_c]
    W_kr: np.ndarray    # [d_model, d_r]
    W_q: np.ndarray     # [d_model, n_h*(d_nope+d_r)]
    W_uk: np.ndarray    # [d_c, n_h*d_nope]
    W_uv: np.ndarray    # [d_c, n_h*d_v]
    W_o: np.ndarray     # [n_h*d_v, d_model]
    raw: dict           # name -> storage array (float32 or uint16 bf16 bits)


def weights(w: Workload) -> Weights:
    shapes = {
        "W_dkv": ((w.d_model, w.d_c), w.d_model),
        "W_kr": ((w.d_model, w.d_r), w.d_model),
        "W_q": ((w.d_model, w.n_h * (w.d_nope + w.d_r)), w.d_model),
        "W_uk": ((w.d_c, w.n_h * w.d_nope), w.d_c),
        "W_uv": ((w.d_c, w.n_h * w.d_v), w.d_c),
        "W_o": ((w.n_h * w.d_v, w.d_model), w.n_h * w.d_v),
    }
    vals, raw = {}, {}
    for k, (name, (shape, fan_in)) in enumerate(shapes.items()):
        a = normal(rng(w.seed, _S_WEIGHTS, k), shape, 1.0 / math.sqrt(fan_in))
        vals[name], raw[name] = to_dtype(a, w.dtype)
    return Weights(raw=raw, **vals)


def seq_lens(w: Workload) -> np.ndarray:
    if w.len_lo == w.len_hi:
        return np.full(w.batch, w.len_lo, dtype=np.int32)
    g = rng(w.seed, _S_LENS)
    return g.integers(w.len_lo, w.len_hi + 1, size=w.batch).astype(np.int32)


def page_table(w: Workload, lens, extra_tokens=0, spare_blocks=0):
    """Shuffled page table with room for max(lens) + extra_tokens per sequence.

    Returns (page_table [B, max_blocks] int32, num_blocks). Sequence b owns
    ceil((lens[b] + extra_tokens) / block_size) distinct blocks drawn from a
    random permutation of all blocks. Entries past a sequence's own blocks
    are -1.
    """
    bs = w.block_size
    need = [(int(L) + extra_tokens + bs - 1) // bs for L in lens]
    max_blocks = max(need) if need else 1
    num_blocks = sum(need) + spare_blocks
    perm = rng(w.seed, _S_PAGES).permutation(num_blocks).astype(np.int32)
    pt = np.full((len(lens), max_blocks), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(need):
        pt[b, :n] = perm[off:off + n]
        off += n
    return pt, num_blocks


def sequence_rows(w: Workload, b, L):
    """Logical cache rows [L, R] of sequence b: (values float32, storage)."""
    a = normal(rng(w.seed, _S_CACHE, b), (int(L), w.R))
    return to_dtype(a, w.dtype)


def fill_paged_cache(w: Workload, lens, pt, num_blocks, fill_value=0.0,
                     keep=None):
    """Paged cache storage [num_blocks, block_size, R] holding every sequence.

    Rows no sequence owns are set to ``fill_value``. Returns (storage array,
    list of per-sequence float32 value arrays). When ``keep`` is a set of
    sequence ids, only those sequences' value arrays are kept (the others are
    None) to save host memory.
    """
    bs = w.block_size
    dt = np.float32 if w.dtype == "f32" else np.uint16
    fill = to_dtype(np.float32([fill_value]), w.dtype)[1][0]
    store = np.full((num_blocks * bs, w.R), fill, dtype=dt)
    vals = [None] * len(lens)
    for b, L in enumerate(lens):
        v, s = sequence_rows(w, b, L)
        if keep is None or b in keep:
            vals[b] = v
        nb = (int(L) + bs - 1) // bs
        for k in range(nb):
            lo, hi = k * bs, min((k + 1) * bs, int(L))
            p = int(pt[b, k])
            store[p * bs:p * bs + (hi - lo)] = s[lo:hi]
    return store.reshape(num_blocks, bs, w.R), vals


def queries(w: Workload):
    """q [B, n_q, n_h, d_nope + d_r] before RoPE: (values float32, storage)."""
    a = normal(rng(w.seed, _S_Q), (w.batch, w.n_q, w.n_h, w.d_nope + w.d_r))
    return to_dtype(a, w.dtype)


def latent_queries(w: Workload):
    """Queries already in latent space, [B, n_q, n_h, d_c + d_r] per head
    [q_lat | q_pe], for the attention core alone: (values float32, storage).
    q_lat ~ N(0, d_nope / d_c), the spread that W_uk^T q_nope has for the
    workloads' weights and queries, and q_pe ~ N(0, 1)."""
    g = rng(w.seed, _S_QLAT)
    shape = (w.batch, w.n_q, w.n_h)
    a = np.concatenate([normal(g, shape + (w.d_c,), math.sqrt(w.d_nope / w.d_c)),
                        normal(g, shape + (w.d_r,))], axis=-1)
    return to_dtype(a, w.dtype)


def hidden_states(w: Workload, T, stream=0):
    """Hidden states x [T, d_model] ~ N(0, 1): (values float32, storage)."""
    a = normal(rng(w.seed, _S_X, stream), (int(T), w.d_model))
    return to_dtype(a, w.dtype)


def fp8_sequence_codes(w: Workload, b, L):
    """Cache rows of sequence b for an fp8 (e4m3) cache, drawn directly as
    codes: (codes uint8 [L, R], row scales float32 [L]).

    Each code byte is assembled from a sign bit, a 4-bit exponent field drawn
    around 12 (magnitudes near 2^5) and a uniform 3-bit mantissa; the NaN
    pattern (exponent 15 with mantissa 7) is never drawn. Row scales are
    uniform in [1/320, 1/96], so the rows' values have a standard deviation
    near one, like the bf16 workloads' rows. No
    rounding or quantisation happens here: both sides decode these bytes.
    """
    g = rng(w.seed, _S_FP8, b)
    L = int(L)
    e = np.clip(np.rint(g.normal(12.0, 2.0, size=(L, w.R))), 0, 15).astype(np.uint8)
    m = g.integers(0, 8, size=(L, w.R), dtype=np.uint8)
    m = np.where((e == 15) & (m == 7), np.uint8(6), m)
    sign = g.integers(0, 2, size=(L, w.R), dtype=np.uint8)
    codes = (sign << 7) | (e << 3) | m
    scales = g.uniform(1 / 320, 1 / 96, size=L).astype(np.float32)
    return codes.astype(np.uint8), scales


def fp8_uniform_codes(w: Workload, b, L):
    """Like fp8_sequence_codes, but every finite e4m3 code (all 254 bytes
    except the two NaN patterns, subnormals and +-448 included) is equally
    likely; row scales uniform in [1/4096, 1/1024]."""
    g = rng(w.seed, _S_FP8, 1000 + b)
    L = int(L)
    c = g.integers(0, 254, size=(L, w.R), dtype=np.int64)
    c = c + (c >= 0x7F) + (c >= 0xFE)   # skip 0x7f and 0xff
    scales = g.uniform(1 / 4096, 1 / 1024, size=L).astype(np.float32)
    return c.astype(np.uint8), scales


def fill_paged_cache_fp8(w: Workload, lens, pt, num_blocks, keep=None):
    """Paged fp8 cache holding every sequence: (codes [num_blocks, bs, R]
    uint8, scales [num_blocks, bs] float32, per-sequence (codes, scales)).
    Rows no sequence owns hold code 0 and scale 0. ``keep`` as for
    fill_paged_cache."""
    bs = w.block_size
    codes = np.zeros((num_blocks * bs, w.R), dtype=np.uint8)
    scales = np.zeros(num_blocks * bs, dtype=np.float32)
    per_seq = [None] * len(lens)
    for b, L in enumerate(lens):
        c, sc = fp8_sequence_codes(w, b, L)
        if keep is None or b in keep:
            per_seq[b] = (c, sc)
        nb = (int(L) + bs - 1) // bs
        for k in range(nb):
            lo, hi = k * bs, min((k + 1) * bs, int(L))
            p = int(pt[b, k])
            codes[p * bs:p * bs + (hi - lo)] = c[lo:hi]
            scales[p * bs:p * bs + (hi - lo)] = sc[lo:hi]
    return codes.reshape(num_blocks, bs, w.R), scales.reshape(num_blocks, bs), per_seq
