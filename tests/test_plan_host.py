"""The split planner on the host (no GPU: okc_plan_options gives the SM count
and the CTAs per SM, so planning makes no CUDA call): every request's visible
keys are covered once, in order, by its work items; item sizes are whole
64-key tiles (counting the TMA-fed tile start of the tcgen05 path); items
launch largest first; the item count respects the waves the heuristic allows;
a list of more than one wave ends in finer items; the plan's sizes agree with
its item list; and the step form follows the documented rule on the
workloads' shapes."""
import numpy as np
import pytest

import fp8_kv_paged_gb300 as okc
import workloads as W

SMS, CTAS = 152, 3  # a GB300 at the q_len-1 decode's occupancy
HOST = {"sm_count": SMS, "ctas_per_sm": CTAS}


@pytest.fixture(scope="module", autouse=True)
def lib():
    okc.build()
    return okc.load()


def _visible(cfg, seq):
    """[lo, hi) of each request's visible keys: the union of its q_len queries'
    windows (all keys up to the block's last on full-attention layers)."""
    L, w = cfg["q_len"], cfg["window"]
    hi = seq.astype(np.int64) + L
    lo = np.maximum(0, seq.astype(np.int64) - w + 1) if w > 0 else np.zeros_like(hi)
    return lo, hi


def _check_cover(cfg, seq, items):
    lo, hi = _visible(cfg, seq)
    B = len(seq)
    by_req = [[] for _ in range(B)]
    for b, j0, j1 in items:
        assert 0 <= b < B and j0 < j1
        by_req[b].append((int(j0), int(j1)))
    for b in range(B):
        by_req[b].sort()  # in key order
        r = by_req[b]
        assert r, f"request {b} has no work item"
        assert r[0][0] == lo[b] and r[-1][1] == hi[b]
        for (a0, a1), (b0, b1) in zip(r, r[1:]):
            assert a1 == b0, f"request {b}: gap or overlap at {a1}/{b0}"
    return by_req


def _pad(cfg, opts=None):
    tc = cfg["q_len"] >= 2 and not ((opts or {}).get("flags", 0) & okc.PLAN_NO_TCGEN05)
    return 7 if tc and cfg["page_size"] >= 8 else 0


@pytest.mark.parametrize("name", list(W.DECODE_WORKLOADS))
def test_workload_plans_cover_every_key_once(name):
    cfg = W.config(name)
    seq = W.lengths(cfg)
    items = okc.okc_attn_plan_items(cfg, seq, HOST)
    by_req = _check_cover(cfg, seq, items)
    sizes = okc.okc_attn_plan_sizes(cfg, seq, HOST)
    assert sizes["num_work"] == len(items)
    assert sizes["max_chunks"] == max(len(r) for r in by_req)
    # launch order: the largest items first
    lens = items[:, 2] - items[:, 1]
    assert np.all(np.diff(lens) <= 0)
    # every item but a request's last holds whole 64-key tiles; within one
    # wave of the resident slots every such item of a request has one size
    pad = _pad(cfg)
    for r in by_req:
        full = {j1 - j0 for j0, j1 in r[:-1]}
        for c in full:
            assert (c + pad) % 64 == 0, c
        if len(items) <= SMS * CTAS:
            assert len(full) <= 1
            if full:
                assert r[-1][1] - r[-1][0] <= max(full)
    # at most four waves of the resident slots (or one item per request)
    assert len(items) <= max(len(seq), 4 * SMS * CTAS)


def test_lists_of_more_than_one_wave_end_in_finer_items():
    """The items that start last decide the step's end, so a q_len-1 list of
    more than one wave of the resident slots ends in smaller items: the mixed
    batch's last tenth of items is at most half the size of its first."""
    cfg = W.config("mixed_full_decode")
    seq = W.lengths(cfg)
    items = okc.okc_attn_plan_items(cfg, seq, HOST)
    assert len(items) > SMS * CTAS
    lens = items[:, 2] - items[:, 1]
    n = len(lens) // 10
    assert lens[-n:].max() * 2 <= lens[:n].min(), (lens[:n].min(), lens[-n:].max())
    # one wave: no item is cut finer than the budget's chunks
    cfg1 = W.config("sliding_decode")
    items1 = okc.okc_attn_plan_items(cfg1, W.lengths(cfg1), HOST)
    assert len(items1) <= SMS * CTAS


def test_step_form_rule_on_the_workloads():
    """One kernel for q_len 1 when the items fill at least half the slots with
    chunks of <= 2048 keys or take more than one wave; else three."""
    want = {"tiny_sliding_decode": 3, "sliding_decode": 1, "full_decode_32k": 3, "verify_block": 3,
            "mixed_full_decode": 1}
    for name, k in want.items():
        cfg = W.config(name)
        seq = W.lengths(cfg)
        assert okc.okc_attn_plan_sizes(cfg, seq, HOST)["step_kernels"] == k, name


@pytest.mark.parametrize("seed", range(12))
def test_random_batches(seed):
    rng = np.random.default_rng(7000 + seed)
    L = int(rng.choice([1, 2, 4, 8]))  # one query block per request (longer ones: _check_blocks)
    P = int(rng.choice([1, 8, 16, 64]))
    window = int(rng.choice([0, 1, 64, 2048]))
    B = int(rng.integers(1, 300))
    seq = rng.integers(0, 40000, size=B).astype(np.int32)
    max_pages = (int(seq.max()) + L + P - 1) // P + 1
    cfg = dict(W.config("tiny_sliding_decode"), batch=B, q_len=L, page_size=P, window=window,
               max_pages=max_pages, num_pages=B * max_pages)
    opts = dict(HOST, ctas_per_sm=int(rng.integers(1, 5)))
    items = okc.okc_attn_plan_items(cfg, seq, opts)
    by_req = _check_cover(cfg, seq, items)
    pad = _pad(cfg)
    for r in by_req:
        if len(r) > 1:
            assert (r[0][1] - r[0][0] + pad) % 64 == 0
    assert len(items) <= max(B, 4 * SMS * opts["ctas_per_sm"])
    # a forced split size is used as given
    forced = okc.okc_attn_plan_items(cfg, seq, dict(opts, chunk_keys=100))
    for r in _check_cover(cfg, seq, forced):
        assert all(j1 - j0 == 100 for j0, j1 in r[:-1])


def test_edge_cases():
    cfg = dict(W.config("tiny_sliding_decode"), batch=3, q_len=8, window=2048, page_size=16,
               max_pages=4, num_pages=12)
    seq = np.array([0, 1, 40], np.int32)
    items = okc.okc_attn_plan_items(cfg, seq, HOST)
    _check_cover(cfg, seq, items)
    assert len(items) == 3  # short requests: one item each
    empty = dict(cfg, batch=0)
    assert len(okc.okc_attn_plan_items(empty, np.zeros(0, np.int32), HOST)) == 0
    # a context past the page table is rejected on the host
    with pytest.raises(okc.OkcError):
        okc.okc_attn_plan_items(cfg, np.array([0, 1, 4 * 16], np.int32), HOST)


def test_items_capacity_and_count_only():
    """count-only query (items NULL, capacity 0), a too-small buffer
    (OKC_ERR_WORKSPACE with the count set), and the exact buffer."""
    import ctypes
    lib = okc.load()
    cfg = W.config("sliding_decode")
    seq = np.ascontiguousarray(W.lengths(cfg), dtype=np.int32)
    c = okc._config(cfg)
    o = okc._options(HOST)
    n = ctypes.c_int32(-1)
    sp = seq.ctypes.data_as(ctypes.c_void_p)
    assert lib.okc_attn_plan_items(ctypes.byref(c), sp, o, None, 0, ctypes.byref(n)) == okc.OK
    total = n.value
    assert total == okc.okc_attn_plan_sizes(cfg, seq, HOST)["num_work"]
    small = np.zeros((total - 1, 3), np.int32)
    n.value = -1
    st = lib.okc_attn_plan_items(ctypes.byref(c), sp, o, small.ctypes.data_as(ctypes.c_void_p), total - 1,
                                 ctypes.byref(n))
    assert st == okc.ERR_WORKSPACE and n.value == total
    full = np.zeros((total, 3), np.int32)
    assert lib.okc_attn_plan_items(ctypes.byref(c), sp, o, full.ctypes.data_as(ctypes.c_void_p), total,
                                   ctypes.byref(n)) == okc.OK
    assert np.array_equal(full, okc.okc_attn_plan_items(cfg, seq, HOST))
    # a null count or a negative capacity is an argument error
    assert lib.okc_attn_plan_items(ctypes.byref(c), sp, o, None, 0, None) == okc.ERR_INVALID
    assert lib.okc_attn_plan_items(ctypes.byref(c), sp, o, None, -1, ctypes.byref(n)) == okc.ERR_INVALID


_SIZE_FIELDS = ("workspace_bytes", "q_fp8_bytes", "o_partial_bytes", "lse_partial_bytes", "num_work", "max_chunks")


def _within_bounds(cfg, seq, opts, max_context):
    bound = okc.okc_attn_plan_max_sizes(cfg, max_context, opts)
    got = okc.okc_attn_plan_sizes(cfg, seq, opts)
    for f in _SIZE_FIELDS:
        assert got[f] <= bound[f], (f, got[f], bound[f])
    assert got["num_tokens"] == bound["num_tokens"]
    return got, bound


@pytest.mark.parametrize("seed", range(16))
def test_max_sizes_bound_every_step(seed):
    """okc_attn_plan_max_sizes bounds okc_attn_plan_sizes for every batch whose
    contexts stay within max_context: random lengths, every request at the
    bound, every request short, forced split sizes, all occupancies."""
    rng = np.random.default_rng(9100 + seed)
    L = int(rng.choice([1, 2, 8, 16]))
    P = int(rng.choice([1, 8, 64]))
    window = int(rng.choice([0, 64, 2048]))
    B = int(rng.choice([1, 7, 64, 300, 1500]))
    max_context = int(rng.integers(L, 140000))
    max_pages = (max_context + P - 1) // P
    cfg = dict(W.config("tiny_sliding_decode"), batch=B, q_len=L, page_size=P, window=window,
               max_pages=max_pages, num_pages=B * max_pages)
    for opts in (dict(HOST, ctas_per_sm=int(rng.integers(1, 5))), dict(HOST, chunk_keys=int(rng.integers(16, 3000)))):
        for seq in (rng.integers(0, max_context - L + 1, size=B),
                    np.full(B, max_context - L),
                    np.minimum(rng.integers(0, 200, size=B), max_context - L)):
            _within_bounds(cfg, seq.astype(np.int32), opts, max_context)


def test_max_sizes_on_the_workloads_and_errors():
    """On each workload's shape the bound holds and is at most four waves of
    items (one per request when requests outnumber them); max_context below
    q_len or past the page table is an argument error."""
    for name in W.DECODE_WORKLOADS:
        cfg = W.config(name)
        seq = W.lengths(cfg)
        max_context = int(seq.max()) + cfg["q_len"]
        _, bound = _within_bounds(cfg, seq, HOST, max_context)
        assert bound["num_work"] <= max(cfg["batch"], 4 * SMS * CTAS)
    cfg = W.config("sliding_decode")
    seq = W.lengths(cfg)  # (sets the page-table shape in cfg)
    for bad in (0, cfg["max_pages"] * cfg["page_size"] + 1):
        with pytest.raises(okc.OkcError) as e:
            okc.okc_attn_plan_max_sizes(cfg, bad, HOST)
        assert e.value.status == okc.ERR_INVALID
    with pytest.raises(okc.OkcError) as e:
        okc.okc_attn_plan_sizes(cfg, seq, dict(HOST, chunk_keys=15))
    assert e.value.status == okc.ERR_INVALID
    empty = dict(cfg, batch=0)
    assert okc.okc_attn_plan_max_sizes(empty, 10, HOST)["num_work"] == 0


def _check_blocks(cfg, seq, ql, items, S):
    """Varlen plans: request b's ql[b] tokens are cut into blocks [i0, i0 + S)
    (the last one shorter), and each block's items cover its visible keys
    [lo, hi) once and in order: hi = seq + i0 + ntok, lo = max(0, seq + i0 - w + 1)
    on window layers, else 0. Requests with no new tokens have no items."""
    w = cfg["window"]
    blocks = {}
    for b, i0, j0, j1 in items:
        assert j0 < j1
        blocks.setdefault((int(b), int(i0)), []).append((int(j0), int(j1)))
    want = set()
    for b, (s0, q) in enumerate(zip(seq.astype(np.int64), ql.astype(np.int64))):
        for i0 in range(0, q, S):
            want.add((b, i0))
            ntok = min(S, q - i0)
            hi = s0 + i0 + ntok
            lo = max(0, s0 + i0 - w + 1) if w > 0 else 0
            r = sorted(blocks[(b, i0)])
            assert r[0][0] == lo and r[-1][1] == hi, (b, i0, r[0], r[-1], lo, hi)
            for (a0, a1), (b0, b1) in zip(r, r[1:]):
                assert a1 == b0
    assert set(blocks) == want


@pytest.mark.parametrize("window", [0, 2048])
@pytest.mark.parametrize("flags,S", [(0, 16), (okc.PLAN_NO_TCGEN05, 16)])
def test_varlen_blocks_cover_every_key_once(window, flags, S):
    """Prefill/extend batches mixing decode requests (1 token), extends of 37,
    256 and 1024 tokens and requests with no new token: blocks of 16 tokens on
    the tcgen05 kernel (its per-KV-head form) and on the warp-level one."""
    rng = np.random.default_rng(window + flags)
    for it in range(20):
        B = int(rng.integers(1, 40))
        cfg = W.config("extend", batch=B, window=window)
        ql = rng.choice([0, 1, 37, 256, 1024], size=B).astype(np.int32)
        seq = rng.integers(0, 20000, size=B).astype(np.int32)
        cfg["max_pages"] = int((seq.max() + 1024) // cfg["page_size"] + 1)
        cfg["num_pages"] = B * cfg["max_pages"]
        opts = dict(HOST, flags=flags)
        items = okc.okc_attn_plan_items_varlen(cfg, seq, ql, opts)
        _check_blocks(cfg, seq, ql, items, S)
        z = okc.okc_attn_plan_sizes(cfg, seq, opts, q_lens=ql)
        assert z["num_work"] == len(items) and z["num_tokens"] == int(ql.sum())
        assert z["o_partial_bytes"] >= len(items) * S * 16 * 64 * 4
        # a uniform q_len of 12 or 40: blocks of S tokens per request, every key covered
        if it == 1:
            for L in (12, 40):
                cu = dict(cfg, q_len=L)
                itm = okc.okc_attn_plan_items_varlen(cu, seq, None, opts)
                _check_blocks(cu, seq, np.full(B, L, np.int32), itm, S)
        # uniform q lengths through the varlen calls: the same plan as without them
        if it == 0:
            u = np.full(B, 3, np.int32)
            c3 = dict(cfg, q_len=3)
            a = okc.okc_attn_plan_items_varlen(c3, seq, u, opts)
            b = okc.okc_attn_plan_items(c3, seq, opts)
            assert np.array_equal(a[:, [0, 2, 3]], b) and np.all(a[:, 1] == 0)


def test_extend_workload_plan():
    cfg = W.config("extend")
    inp = W.generate(cfg)
    items = okc.okc_attn_plan_items_varlen(cfg, inp["seq_lens"], inp["q_lens"], {"sm_count": SMS, "ctas_per_sm": 1})
    _check_blocks(cfg, inp["seq_lens"], inp["q_lens"], items, 16)
    bound = okc.okc_attn_plan_max_sizes(cfg, int((inp["seq_lens"] + inp["q_lens"]).max()),
                                        {"sm_count": SMS, "ctas_per_sm": 1})
    z = okc.okc_attn_plan_sizes(cfg, inp["seq_lens"], {"sm_count": SMS, "ctas_per_sm": 1}, q_lens=inp["q_lens"])
    for f in ("workspace_bytes", "o_partial_bytes", "num_work", "q_fp8_bytes"):
        assert z[f] <= bound[f], f


def test_fixed_capacity_plans_keep_their_layout():
    """okc_plan_options.max_context: the workspace is laid out at the capacity
    of okc_attn_plan_max_sizes for that context, for every step within it; steps
    past it and per-request q lengths are refused."""
    for name in W.DECODE_WORKLOADS:
        cfg = W.config(name)
        seq = W.lengths(cfg)
        mc = int(seq.max()) + cfg["q_len"]
        opts = dict(HOST, max_context=mc)
        bound = okc.okc_attn_plan_max_sizes(cfg, mc, opts)
        for s in (seq, np.minimum(seq, 7), seq // 2):
            z = okc.okc_attn_plan_sizes(cfg, s, opts)
            assert z["workspace_bytes"] == bound["workspace_bytes"], name
            assert z["num_work"] == okc.okc_attn_plan_sizes(cfg, s, HOST)["num_work"]
        with pytest.raises(okc.OkcError) as e:
            okc.okc_attn_plan_sizes(cfg, seq + 1, opts)
        assert e.value.status == okc.ERR_INVALID
        with pytest.raises(okc.OkcError) as e:
            okc.okc_attn_plan_sizes(cfg, seq, opts, q_lens=np.full(len(seq), cfg["q_len"], np.int32))
        assert e.value.status == okc.ERR_UNSUPPORTED
