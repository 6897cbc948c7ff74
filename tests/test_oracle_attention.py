"""Pins of the oracle's step 4 (the flash_attn_with_kvcache call of the Muse
Spark attention problem file: paged, causal, window_size (window-1, 0)) and of
step 5 (rms_norm_gate): a dense brute force written from the definition in
numpy, and the invariances the page fixes (window edge, causality inside the
verify block, page-table permutation), plus closed forms of the norm-gate.
"""
import numpy as np
import pytest

import oracle
import workloads as W

HQ, HKV, D = 16, 2, 64


def _tiny(L=1, P=1, window=0, seq=(5, 11), kv_scale=1.0, seed=0):
    cfg = W.config("tiny_sliding_decode", batch=len(seq), q_len=L, page_size=P, window=window,
                   seq=("list", list(seq)), kv_scale=kv_scale, rope_theta=5e5, seed=seed)
    inp = W.generate(cfg)
    return cfg, inp


def _dense_reference(cfg, inp, q8, k_cache, v_cache):
    """Dense softmax attention from the definition: gather each request's keys
    0..n-1 into a matrix, build the mask matrix, softmax row by row."""
    L, P, w = cfg["q_len"], cfg["page_size"], cfg["window"]
    ks = float(inp["k_scale"]) if cfg["kv_scale"] != 1.0 else 1.0
    vs = float(inp["v_scale"]) if cfg["kv_scale"] != 1.0 else 1.0
    if cfg.get("q_norm", 0) == 1:  # the factor is inside q (the vLLM qk_norm with an output scale)
        scale = float(np.float32(cfg["sm_scale"]))
    else:
        scale = float(np.float32(cfg["sm_scale"] * cfg["qk_scale_factor"]))
    kc = k_cache.reshape(-1, HKV, D)
    vc = v_cache.reshape(-1, HKV, D)
    out = np.zeros((q8.shape[0], HQ, D))
    lse = np.zeros((q8.shape[0], HQ))
    # request b's new tokens: rows t0 .. t0 + ql - 1 (ql = L each unless q_lens says otherwise)
    q_lens = inp.get("q_lens") if "q_lens" in cfg else None
    t0 = 0
    for b in range(cfg["batch"]):
        ql = L if q_lens is None else int(q_lens[b])
        n = int(inp["cache_seqlens"][b])
        rows = [inp["page_table"][b, j // P] * P + j % P for j in range(n)]
        K = oracle.e4m3_value(kc[rows]) * ks          # [n, Hkv, D]
        V = oracle.e4m3_value(vc[rows]) * vs
        pos = n - ql + np.arange(ql)                  # query positions
        j = np.arange(n)
        allowed = j[None, :] <= pos[:, None]
        if w > 0:
            allowed &= j[None, :] >= pos[:, None] - w + 1
        t_first, t0 = t0, t0 + ql
        for i in range(ql):
            t = t_first + i
            Q = oracle.e4m3_value(q8[t])              # [Hq, D]
            for h in range(HQ):
                g = h // (HQ // HKV)
                s = (K[:, g, :] @ Q[h]) * scale
                s = np.where(allowed[i], s, -np.inf)
                m = s.max()
                e = np.exp(s - m)
                out[t, h] = (e @ V[:, g, :]) / e.sum()
                lse[t, h] = m + np.log(e.sum())
    return out, lse


@pytest.mark.parametrize("L,P,window,seq,kv_scale", [
    (1, 1, 0, (5, 11), 1.0),
    (1, 1, 4, (0, 9), 1.0),
    (8, 1, 0, (3, 7), 1.0),
    (8, 4, 5, (0, 13), 0.5),
    (1, 4, 3, (6, 16), 0.5),
])
def test_matches_dense_brute_force(L, P, window, seq, kv_scale, q_norm=0):
    cfg, inp = _tiny(L=L, P=P, window=window, seq=seq, kv_scale=kv_scale)
    cfg["q_norm"] = q_norm
    if kv_scale != 1.0:
        inp["k_scale"] = np.float32(kv_scale)
        inp["v_scale"] = np.float32(kv_scale * 1.5)
    k = inp["k_cache"].copy(); v = inp["v_cache"].copy()
    q8, _ = oracle.prepare(cfg, inp, k, v)
    o, lse, bad = oracle.attention(cfg, inp, q8, k, v, want_lse=True)
    ref, ref_lse = _dense_reference(cfg, inp, q8, k, v)
    assert bad == 0
    assert np.max(np.abs(o - ref)) < 1e-12
    assert np.max(np.abs(lse - ref_lse)) < 1e-10


@pytest.mark.parametrize("window", [0, 4])
def test_ragged_batch_matches_dense_brute_force(window):
    """Per-request q lengths (ragged cu_seqlens_q, a request with none among
    them): each request's tokens at rows cu_seqlens_q[b].., causal over its
    own earlier keys; equal to the dense definition."""
    cfg = W.config("tiny_sliding_decode", batch=4, q_len=6, q_lens=("list", [3, 0, 6, 1]), page_size=2,
                   window=window, seq=("list", [5, 2, 0, 9]), rope_theta=5e5)
    inp = W.generate(cfg)
    assert list(inp["cu_seqlens_q"]) == [0, 3, 3, 9, 10]
    k = inp["k_cache"].copy(); v = inp["v_cache"].copy()
    q8, _ = oracle.prepare(cfg, inp, k, v)
    o, lse, bad = oracle.attention(cfg, inp, q8, k, v, want_lse=True)
    ref, ref_lse = _dense_reference(cfg, inp, q8, k, v)
    assert bad == 0
    assert np.max(np.abs(o - ref)) < 1e-12
    assert np.max(np.abs(lse - ref_lse)) < 1e-10


def test_folded_q_norm_matches_dense_brute_force():
    """q_norm 1: the softmax scale is sm_scale alone (the factor is inside q)."""
    test_matches_dense_brute_force(8, 4, 5, (0, 13), 0.5, q_norm=1)
    test_matches_dense_brute_force(1, 1, 0, (5, 11), 1.0, q_norm=1)


def test_folded_q_norm_computes_the_same_block():
    """Both q norms compute the same attention up to the E4M3 rounding of q: the
    logits q.k * scale agree within the quantisation of q (the factor moved from
    the scale into q), and the block's outputs agree to within that noise."""
    for seq, L, w in (((300, 2100, 40), 1, 2048), ((500, 900), 8, 0)):
        cfg = W.config("tiny_sliding_decode", batch=len(seq), q_len=L, window=w, seq=("list", list(seq)))
        inp = W.generate(cfg)
        a = oracle.step(dict(cfg, q_norm=0), inp)
        b = oracle.step(dict(cfg, q_norm=1), inp)
        qa = oracle.e4m3_value(a["q8"]) * cfg["qk_scale_factor"]
        qb = oracle.e4m3_value(b["q8"])
        # each E4M3 value is within 1/16 relative of what it rounds, so |qa - qb| <=
        # (1/8) / (15/16) of the larger, plus the absolute error of the rotation
        # (its bf16 roundings are relative to the pair's norm, ~3 * 2^-9 * 5.473)
        assert np.all(np.abs(qa - qb) <= (2.0 / 15.0) * np.maximum(np.abs(qa), np.abs(qb)) + 0.05)
        oa = oracle.bf16_value(a["out"])
        ob = oracle.bf16_value(b["out"])
        err = np.abs(oa - ob)
        assert err.mean() < 0.05 and np.corrcoef(oa.ravel(), ob.ravel())[0, 1] > 0.985, (err.mean(), err.max())


def _attend(cfg, inp, k, v, q8):
    o, _ = oracle.attention(cfg, inp, q8, k, v)
    return o


def test_window_keeps_token_and_2047_before_it():
    cfg, inp = _tiny(window=2048, seq=(3000, 2500))
    k = inp["k_cache"].copy(); v = inp["v_cache"].copy()
    q8, _ = oracle.prepare(cfg, inp, k, v)
    base = _attend(cfg, inp, k, v, q8)
    P = cfg["page_size"]
    p = int(inp["positions"][0])                      # query position of request 0
    for j, expect_change in ((p - 2048, False), (p - 2047, True)):
        k2, v2 = k.copy(), v.copy()
        row = inp["page_table"][0, j // P] * P + j % P
        k2.reshape(-1, HKV * D)[row] ^= 0x11
        v2.reshape(-1, HKV * D)[row] ^= 0x11
        o2 = _attend(cfg, inp, k2, v2, q8)
        changed = not np.array_equal(o2[0], base[0])
        assert changed == expect_change, j
        assert np.array_equal(o2[1], base[1])         # the other request never moves


def test_wide_window_equals_full_attention():
    cfg, inp = _tiny(window=0, seq=(40, 70))
    k = inp["k_cache"].copy(); v = inp["v_cache"].copy()
    q8, _ = oracle.prepare(cfg, inp, k, v)
    full = _attend(cfg, inp, k, v, q8)
    wide = _attend(dict(cfg, window=71), inp, k, v, q8)
    assert np.array_equal(full, wide)
    narrow = _attend(dict(cfg, window=70), inp, k, v, q8)
    assert not np.array_equal(full[1], narrow[1]) and np.array_equal(full[0], narrow[0])


def test_page_table_permutation_invariance():
    cfg, inp = _tiny(P=4, seq=(37, 50))
    k = inp["k_cache"].copy(); v = inp["v_cache"].copy()
    q8, _ = oracle.prepare(cfg, inp, k, v)
    base = _attend(cfg, inp, k, v, q8)
    rng = np.random.default_rng(9)
    perm = rng.permutation(cfg["num_pages"])          # new physical id of page p
    k2 = np.empty_like(k); v2 = np.empty_like(v)
    k2[perm] = k; v2[perm] = v
    pt = inp["page_table"].copy()
    pt[pt >= 0] = perm[pt[pt >= 0]]
    o2 = _attend(cfg, dict(inp, page_table=pt), k2, v2, q8)
    assert np.array_equal(o2, base)


def test_verify_block_is_causal():
    cfg, inp = _tiny(L=8, seq=(20, 33))
    k = inp["k_cache"].copy(); v = inp["v_cache"].copy()
    q8, _ = oracle.prepare(cfg, inp, k, v)
    base = _attend(cfg, inp, k, v, q8)
    P = cfg["page_size"]
    for i in range(7):
        # disturb the cache row of block token i+1 of request 1
        j = int(inp["positions"][8 + i + 1])
        row = inp["page_table"][1, j // P] * P + j % P
        k2 = k.copy(); k2.reshape(-1, HKV * D)[row] ^= 0x22
        o2 = _attend(cfg, inp, k2, v, q8)
        assert np.array_equal(o2[8:8 + i + 1], base[8:8 + i + 1])   # queries <= i unchanged
        assert not np.array_equal(o2[8 + i + 1], base[8 + i + 1])
        assert np.array_equal(o2[:8], base[:8])


def test_empty_history_request():
    """seq_len 0 (a padded slot): the query sees only its own new key, so its
    output is that key's value row for every head of the group."""
    cfg, inp = _tiny(seq=(0, 4))
    k = inp["k_cache"].copy(); v = inp["v_cache"].copy()
    q8, _ = oracle.prepare(cfg, inp, k, v)
    o = _attend(cfg, inp, k, v, q8)
    row = int(inp["cache_loc"][0])
    vrow = oracle.e4m3_value(v.reshape(-1, HKV, D)[row])
    for h in range(HQ):
        assert np.array_equal(o[0, h], vrow[h // 8])


def test_lse_merge_of_key_splits():
    """Splitting a request's keys into chunks and merging the chunk outputs by
    log-sum-exp reproduces the unsplit output (the identity split-KV relies on)."""
    cfg, inp = _tiny(seq=(60, 90))
    k = inp["k_cache"].copy(); v = inp["v_cache"].copy()
    q8, _ = oracle.prepare(cfg, inp, k, v)
    o, lse, _ = oracle.attention(cfg, inp, q8, k, v, want_lse=True)
    # chunk outputs via windows: keys [p-w+1, p] minus keys [p-w'+1, p] is a chunk;
    # use the dense reference on masked chunks instead
    ref, _ = _dense_reference(cfg, inp, q8, k, v)
    kc = oracle.e4m3_value(k.reshape(-1, HKV, D)); vc = oracle.e4m3_value(v.reshape(-1, HKV, D))
    if cfg.get("q_norm", 0) == 1:  # the factor is inside q (the vLLM qk_norm with an output scale)
        scale = float(np.float32(cfg["sm_scale"]))
    else:
        scale = float(np.float32(cfg["sm_scale"] * cfg["qk_scale_factor"]))
    b, t = 1, 1
    n = int(inp["cache_seqlens"][b])
    rows = inp["page_table"][b, :n]
    for h in (0, 9):
        g = h // 8
        s = (kc[rows, g] @ oracle.e4m3_value(q8[t, h])) * scale
        parts = []
        for lo, hi in ((0, 17), (17, 64), (64, n)):
            m = s[lo:hi].max(); e = np.exp(s[lo:hi] - m)
            parts.append((m + np.log(e.sum()), (e @ vc[rows[lo:hi], g]) / e.sum()))
        L_ = np.logaddexp.reduce([p[0] for p in parts])
        merged = sum(np.exp(p[0] - L_) * p[1] for p in parts)
        assert np.max(np.abs(merged - o[t, h])) < 1e-12
        assert abs(L_ - lse[t, h]) < 1e-12


# ------------------------------------------------------------------ norm-gate

def _normgate_case(o, gate_vals, weight=None):
    cfg, inp = _tiny(seq=(3, 4))
    qkv = inp["qkv"].copy()
    gcol = (HQ + 2 * HKV) * D
    qkv[:, gcol:] = oracle.bf16_bits(np.broadcast_to(gate_vals, (qkv.shape[0], HQ * D)))
    return oracle.bf16_value(oracle.normgate(cfg, o, qkv, weight, 1e-5))


def test_normgate_saturated_gate_is_plain_rmsnorm():
    rng = np.random.default_rng(4)
    o = rng.standard_normal((2, HQ, D))
    w = W._bf16_bits(1 + 0.1 * rng.standard_normal(D))
    got = _normgate_case(o, 80.0, w).reshape(2, HQ, D)        # sigmoid(80) == 1 in double
    ob = oracle.bf16_value(oracle.bf16_bits(o))
    rms = np.sqrt((ob ** 2).mean(axis=2, keepdims=True) + 1e-5)
    ref = ob / rms * oracle.bf16_value(w)
    assert np.max(np.abs(got - ref) / np.maximum(np.abs(ref), 1e-3)) <= 2.0 ** -8


def test_normgate_constant_head_and_zero_gate():
    o = np.zeros((2, HQ, D))
    o[:, :, :] = np.linspace(-3, 3, HQ)[None, :, None]       # constant within each head
    got = _normgate_case(o, 0.0).reshape(2, HQ, D)           # sigmoid(0) = 1/2
    ob = oracle.bf16_value(oracle.bf16_bits(o))
    ref = np.sign(ob) * np.abs(ob) / np.sqrt(ob ** 2 + 1e-5) * 0.5
    assert np.max(np.abs(got - ref)) <= 2.0 ** -9
    assert np.all(np.abs(got[np.abs(o) > 0.1]) - 0.5 <= 2.0 ** -9)


def test_normgate_weight_none_equals_ones():
    rng = np.random.default_rng(6)
    o = rng.standard_normal((2, HQ, D))
    g = rng.standard_normal(HQ * D)
    ones = oracle.bf16_bits(np.ones(D))
    assert np.array_equal(_normgate_case(o, g, None), _normgate_case(o, g, ones))
