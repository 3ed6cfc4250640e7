"""bench.py's roofline accounting, checked on CPU.

The attention kernel's algorithmic work per decode call is one cache row
(d_c + d_r elements) per cached token, and 2 * n_h * (R + d_c) FLOPs per
visible (row, query) pair: the score against [c | k_rope] (R wide) and the
weighted sum of c (d_c wide), for every head. Query i of a sequence of
length L sees L - n_q + i + 1 rows.
"""
import numpy as np

import bench
from mla_latent_kv_73_b300 import synth


def test_dsv2_batch16_figures():
    w = synth.WORKLOADS["dsv2_b16_l4096"]
    lens = synth.seq_lens(w)
    assert np.all(lens == 4096) and len(lens) == 16
    cache_bytes, flops = bench.algorithmic(w, lens)
    assert cache_bytes == 16 * 4096 * 1152 == 75_497_472
    assert flops == 2 * 128 * (576 + 512) * 16 * 4096
    assert round(flops / 1e9, 2) == 18.25
    # the HBM roofline time at the measured copy rate
    assert abs(cache_bytes / 6514.2e9 * 1e6 - 11.59) < 0.01


def test_two_query_tokens_see_causal_rows():
    w = synth.WORKLOADS["dsv2_b4_l131072_nq2"]
    lens = synth.seq_lens(w)
    cache_bytes, flops = bench.algorithmic(w, lens)
    assert cache_bytes == 4 * 131072 * 1152 and round(cache_bytes / 1e6, 2) == 603.98
    visible = 4 * ((131072 - 2 + 0 + 1) + (131072 - 2 + 1 + 1))
    assert flops == 2 * 128 * 1088 * visible and round(flops / 1e9, 2) == 292.06
    # two queries per row: twice the FLOPs per cache byte of one query, so
    # the tensor pipe bounds this one at the measured bf16 rate
    assert flops / 1786.4e12 > cache_bytes / 6514.2e9


def test_ragged_workloads_by_brute_force():
    for name in ("dsv2_b64_ragged", "nh16_b256_ragged"):
        w = synth.WORKLOADS[name]
        lens = synth.seq_lens(w)
        cache_bytes, flops = bench.algorithmic(w, lens)
        rows = vis = 0
        for L in lens:
            for j in range(int(L)):
                rows += 1
            for i in range(w.n_q):
                vis += int(L) - w.n_q + i + 1
        assert cache_bytes == rows * w.R * 2
        assert flops == 2.0 * w.n_h * (w.R + w.d_c) * vis


def test_whole_step_bytes_and_flops():
    """The whole step's roofline counts every input and output once: the
    cache, the append's W_dkv||W_kr, W_uk and W_uv (bf16), the new tokens'
    hidden states and rows, the queries, and the fp32 output."""
    w = synth.WORKLOADS["dsv2_b16_l4096"]
    lens = synth.seq_lens(w)
    nbytes, flops = bench.step_algorithmic(w, lens)
    tensors = {
        "cache": 16 * 4096 * 576 * 2,
        "W_dkv||W_kr": 5120 * 576 * 2,
        "W_uk": 512 * 128 * 128 * 2,
        "W_uv": 512 * 128 * 128 * 2,
        "x": 16 * 5120 * 2,
        "new rows": 16 * 576 * 2,
        "q": 16 * 128 * 192 * 2,
        "out": 16 * 128 * 128 * 4,
    }
    assert nbytes == sum(tensors.values()) == 116_967_424
    _, attn = bench.algorithmic(w, lens)
    assert flops == attn + 2 * 16 * (5120 * 576 + 128 * 512 * 128 * 2)
    r = bench.roofline_entry(nbytes, flops, 0.0666, 6514.2, 1786.4)
    assert r["bound"] == "hbm" and abs(r["frac"] - nbytes / 66.6e-6 / 6514.2e9) < 1e-4
