"""The seeded input recipe: each workload's generated step has the structure
the recipe states — every request's pages distinct physical pages of a pool of
exactly the total size, -1 past its pages; positions seq + i; cache_loc the
flat row of each position through the page table; cache_seqlens seq + L;
cu_seqlens_q 0, L, 2L, ...; lengths within the recipe's range; qkv of the
2304-wide layout; E4M3 cache fill without NaN codes — and lengths() draws the
same lengths as generate() without building the caches."""
import numpy as np
import pytest

import workloads as W

SMALL = {"tiny_sliding_decode": {}, "sliding_decode": dict(batch=16), "full_decode_32k": dict(batch=3, seq=("const", 700)),
         "verify_block": dict(batch=6), "mixed_full_decode": dict(batch=40, seq=("loguniform", 1, 5000)),
         "extend": dict(batch=12, seq=("uniform", 0, 3000))}


@pytest.mark.parametrize("name", list(W.WORKLOADS))
def test_generated_step_has_the_recipes_structure(name):
    cfg = W.config(name, **SMALL[name])
    inp = W.generate(cfg)
    B, L, P = cfg["batch"], cfg["q_len"], cfg["page_size"]
    seq = inp["seq_lens"].astype(np.int64)
    kind = cfg["seq"][0]
    if kind == "uniform" or kind == "loguniform":
        assert seq.min() >= cfg["seq"][1] and seq.max() <= cfg["seq"][2]
    elif kind == "const":
        assert (seq == cfg["seq"][1]).all()
    else:
        assert list(seq) == list(cfg["seq"][1])
    ql = inp["q_lens"].astype(np.int64)  # new tokens per request (L each, or the "q_lens" recipe)
    if "q_lens" in cfg:
        assert set(ql) <= set(cfg["q_lens"][1]) and ql.max() <= L
    else:
        assert (ql == L).all()
    n_pages = (seq + ql + P - 1) // P
    pt = inp["page_table"]
    assert pt.shape == (B, n_pages.max()) and cfg["num_pages"] == n_pages.sum()
    used = np.concatenate([pt[b, :n_pages[b]] for b in range(B)])
    assert np.array_equal(np.sort(used), np.arange(n_pages.sum()))  # a permutation of the pool
    for b in range(B):
        assert (pt[b, n_pages[b]:] == -1).all()
    T = int(ql.sum())
    cu = np.concatenate([[0], np.cumsum(ql)])
    for b in range(B):
        assert np.array_equal(inp["positions"][cu[b]:cu[b + 1]], seq[b] + np.arange(ql[b]))
    req = np.repeat(np.arange(B), ql)
    p = inp["positions"]
    assert np.array_equal(inp["cache_loc"], pt[req, p // P].astype(np.int64) * P + p % P)
    assert np.array_equal(inp["cache_seqlens"], seq + ql)
    assert np.array_equal(inp["cu_seqlens_q"], cu)
    if "q_lens" not in cfg:
        assert np.array_equal(inp["cu_seqlens_q"], np.arange(B + 1) * L)
    assert inp["qkv"].shape == (T, 2304) and inp["qkv"].dtype == np.uint16
    assert inp["k_cache"].shape == (n_pages.sum(), P, 2, 64) and inp["k_cache"].dtype == np.uint8
    for c in (inp["k_cache"], inp["v_cache"]):
        assert not np.isin(c, [0x7F, 0xFF]).any()  # no E4M3 NaN codes in the fill
    assert float(inp["k_scale"]) == cfg["kv_scale"]
    assert (inp["norm_weight"] is None) == (not cfg["norm_weight"])


@pytest.mark.parametrize("name", list(W.WORKLOADS))
def test_lengths_match_generate(name):
    a, b = W.config(name, **SMALL[name]), W.config(name, **SMALL[name])
    seq = W.lengths(a)
    inp = W.generate(b)
    assert np.array_equal(seq, inp["seq_lens"])
    assert (a["max_pages"], a["num_pages"]) == (b["max_pages"], b["num_pages"])


def test_full_size_lengths():
    """The full-size recipes: sliding U[1024, 8192]; verify U[8192, 16384]; the
    mixed batch floor(exp(U(0, ln 131072))) within [1, 131072] with a median
    near sqrt(131072)."""
    s = W.lengths(W.config("sliding_decode"))
    assert len(s) == 64 and s.min() >= 1024 and s.max() <= 8192
    v = W.lengths(W.config("verify_block"))
    assert len(v) == 32 and v.min() >= 8192 and v.max() <= 16384
    m = W.lengths(W.config("mixed_full_decode"))
    assert len(m) == 256 and m.min() >= 1 and m.max() <= 131072
    assert 100 < np.median(m) < 3000
