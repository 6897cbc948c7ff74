"""GPU parity of okc_attn_step, the whole block in one launch: against the
oracle under the acceptance bounds, and bit for bit against the three-call
path (same arithmetic, same merge order), on the workloads' shapes, edge cases
and forced split counts; consecutive launches reuse the plan's arrival counters."""
import numpy as np
import pytest

import workloads as W
from parity_util import check_against_oracle, full_check, run_gpu, to_device
from test_gpu_parity import SMALL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib):
    return cuda_lib


def _same_as_three_call(cfg, inp, opts=None):
    a = run_gpu(cfg, inp, opts)
    b = run_gpu(cfg, inp, opts, fused=True)
    assert b["errors"] == 0
    assert np.array_equal(a["out"], b["out"])
    assert np.array_equal(a["k_cache"], b["k_cache"]) and np.array_equal(a["v_cache"], b["v_cache"])


@pytest.mark.parametrize("name", list(SMALL))
def test_fused_workload_shapes(name):
    cfg = W.config(name, **SMALL[name])
    inp = W.generate(cfg)
    rep = full_check(cfg, inp, fused=True)
    print(name, rep)
    _same_as_three_call(cfg, inp)


@pytest.mark.parametrize("chunk", [16, 100, 100000])
@pytest.mark.parametrize("name", ["sliding_decode", "verify_block"])
def test_fused_forced_splits(name, chunk):
    cfg = W.config(name, **SMALL[name])
    inp = W.generate(cfg)
    full_check(cfg, inp, opts={"chunk_keys": chunk}, fused=True)
    _same_as_three_call(cfg, inp, {"chunk_keys": chunk})


@pytest.mark.parametrize("seq,L,window,P", [
    ([0, 1, 2, 3], 1, 2048, 1),
    ([0, 5, 70, 129], 8, 2048, 64),
    ([2046, 2047, 2048, 2049], 1, 2048, 1),
    ([2040, 2041, 2047, 2055], 8, 2048, 1),
    ([300, 17, 1000], 4, 256, 16),
    ([900, 33], 16, 512, 256),
])
def test_fused_edge_shapes(seq, L, window, P):
    cfg = W.config("tiny_sliding_decode", batch=len(seq), q_len=L, window=window, page_size=P,
                   seq=("list", seq))
    inp = W.generate(cfg)
    full_check(cfg, inp, fused=True)
    full_check(cfg, inp, opts={"chunk_keys": 32}, fused=True)


def test_fused_repeated_launches_reuse_tickets():
    import fp8_kv_paged_gb300 as okc
    import torch
    cfg = W.config("sliding_decode", batch=6, seq=("uniform", 1500, 2600))
    inp = W.generate(cfg)
    d = to_device(cfg, inp)
    step = okc.AttnStep(cfg, inp["seq_lens"], opts={"chunk_keys": 256, "flags": okc.PLAN_STEP_ONE_LAUNCH})
    assert step.sizes["step_kernels"] == 1
    outs = []
    for _ in range(3):
        outs.append(step.run_fused(d, eps=inp["eps"]).clone())
    torch.cuda.synchronize()
    assert step.errors() == 0
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


def test_step_form_chosen_by_the_plan():
    """q_len 1 steps that fill the GPU with short chunks run as one kernel; very
    small batches, long chunks and verify blocks as three; the flags override
    (verify blocks of up to 8 tokens on the tcgen05 kernel have a one-kernel
    form too; longer blocks and the warp-level kernel do not)."""
    import fp8_kv_paged_gb300 as okc
    sliding = W.config("sliding_decode")
    seq = W.generate(sliding)["seq_lens"]
    assert okc.okc_attn_plan_sizes(sliding, seq)["step_kernels"] == 1
    assert okc.okc_attn_plan_sizes(sliding, seq, {"flags": okc.PLAN_STEP_THREE_LAUNCHES})["step_kernels"] == 3
    tiny = W.config("tiny_sliding_decode")
    tseq = W.generate(tiny)["seq_lens"]
    assert okc.okc_attn_plan_sizes(tiny, tseq)["step_kernels"] == 3
    assert okc.okc_attn_plan_sizes(tiny, tseq, {"flags": okc.PLAN_STEP_ONE_LAUNCH})["step_kernels"] == 1
    full = dict(W.config("full_decode_32k"), max_pages=32769, num_pages=64 * 32769)
    assert okc.okc_attn_plan_sizes(full, np.full(64, 32768, np.int32))["step_kernels"] == 3  # one wave, long chunks
    mixed = W.config("mixed_full_decode")
    mseq = W.generate(mixed)["seq_lens"]
    msz = okc.okc_attn_plan_sizes(mixed, mseq)
    assert msz["step_kernels"] == 1 and msz["num_work"] > 456  # more than one wave
    verify = W.config("verify_block")
    vseq = W.generate(verify)["seq_lens"]
    assert okc.okc_attn_plan_sizes(verify, vseq)["step_kernels"] == 3
    # blocks of 2..8 tokens on the tcgen05 kernel: one kernel when asked for
    assert okc.okc_attn_plan_sizes(verify, vseq, {"flags": okc.PLAN_STEP_ONE_LAUNCH})["step_kernels"] == 1
    warp = {"flags": okc.PLAN_STEP_ONE_LAUNCH | okc.PLAN_NO_TCGEN05}
    assert okc.okc_attn_plan_sizes(verify, vseq, warp)["step_kernels"] == 3
    longer = dict(verify, q_len=12)
    assert okc.okc_attn_plan_sizes(longer, vseq, {"flags": okc.PLAN_STEP_ONE_LAUNCH})["step_kernels"] == 3


def _host_tensor(a, memory):
    """A host tensor holding `a`: pinned, pageable, or pinned at an address one
    element past an aligned allocation (misaligned for 16-byte vectors)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    if memory == "pageable":
        return t.clone()
    if memory == "pinned":
        return t.pin_memory()
    flat = torch.empty(t.numel() + 1, dtype=t.dtype).pin_memory()
    view = flat[1:].view(t.shape)
    view.copy_(t)
    return view


@pytest.mark.parametrize("memory", ["pinned", "pageable", "pinned_offset"])
@pytest.mark.parametrize("name", ["sliding_decode", "verify_block", "full_decode_32k"])
def test_step_from_host_buffers(name, memory):
    """okc_attn_step_host: host inputs copied in (one gather kernel for
    device-mapped pinned buffers, at any alignment; the copy engine for
    pageable ones), the step, the output copied back: equal to okc_attn_step on
    device buffers, bit for bit."""
    import fp8_kv_paged_gb300 as okc
    import torch
    from test_gpu_parity import SMALL
    cfg = W.config(name, **SMALL[name])
    inp = W.generate(cfg)
    d = to_device(cfg, inp)
    ref = run_gpu(cfg, inp, fused=True, plan_form=True)
    step = okc.AttnStep(cfg, inp["seq_lens"])
    host = {k: _host_tensor(inp[k], memory)
            for k in ("positions", "cache_loc", "cache_seqlens", "cu_seqlens_q", "seq_lens", "page_table")}
    host["qkv"] = _host_tensor(np.ascontiguousarray(inp["qkv"]).view(np.int16), memory)
    host["out"] = _host_tensor(np.zeros((inp["qkv"].shape[0], 1024), np.int16), memory)
    dev = {k: torch.empty_like(v, device="cuda") for k, v in host.items()}
    okc.okc_attn_step_host(step.plan, host, dev, d["k_cache"], d["v_cache"], d["k_scale"], d["v_scale"],
                           d.get("rope_table"), d["norm_weight"], inp["eps"], step.o_partial, step.lse_partial)
    assert step.errors() == 0
    assert np.array_equal(host["out"].numpy().view(np.uint16), ref["out"])
    assert np.array_equal(d["k_cache"].cpu().numpy(), ref["k_cache"])
    check_against_oracle(cfg, inp, host["out"].numpy().view(np.uint16), d["k_cache"].cpu().numpy(),
                         d["v_cache"].cpu().numpy())


@pytest.mark.parametrize("name", ["sliding_decode", "verify_block", "tiny_sliding_decode"])
def test_step_replays_from_a_cuda_graph(name):
    """okc_attn_step captured in a CUDA graph and replayed after the caller
    rewrote its input buffers (new qkv, new cache contents, same lengths) gives
    the eager result for the new contents, bit for bit: the kernels read every
    input and length from device memory when they run."""
    import fp8_kv_paged_gb300 as okc
    import torch
    from test_gpu_parity import SMALL
    cfg = W.config(name, **SMALL[name])
    inp = W.generate(cfg)
    other = W.generate(dict(cfg), seed=cfg["seed"] + 101)
    inp2 = dict(inp, qkv=other["qkv"], k_cache=np.roll(inp["k_cache"], 3), v_cache=np.roll(inp["v_cache"], 5))
    d = to_device(cfg, inp)
    step = okc.AttnStep(cfg, inp["seq_lens"])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step.run_fused(d, eps=inp["eps"], stream=s)  # warm the launch path
    s.synchronize()
    d = to_device(cfg, inp)  # fresh caches: the warm-up wrote the new rows
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step.run_fused(d, eps=inp["eps"], stream=s)
    for case in (inp, inp2):
        fresh = to_device(cfg, case)
        for k in ("qkv", "k_cache", "v_cache"):
            d[k].copy_(fresh[k])
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        got_out = step.out.view(torch.int16).cpu().numpy().view(np.uint16)
        got_k = d["k_cache"].cpu().numpy()
        ref = run_gpu(cfg, case, plan_form=True, fused=True)
        assert step.errors() == 0
        assert np.array_equal(got_out, ref["out"])
        assert np.array_equal(got_k, ref["k_cache"])
        check_against_oracle(cfg, case, got_out, got_k, d["v_cache"].cpu().numpy())


def _shorter(cfg, inp, d):
    """The same batch d tokens earlier: every context d keys shorter (same
    caches and page table, positions and cache rows moved back)."""
    out = dict(inp)
    out["seq_lens"] = inp["seq_lens"] - d
    out["cache_seqlens"] = inp["cache_seqlens"] - d
    out["positions"] = inp["positions"] - d
    P, L = cfg["page_size"], cfg["q_len"]
    req = np.repeat(np.arange(cfg["batch"]), L)
    pos = out["positions"]
    out["cache_loc"] = inp["page_table"][req, pos // P].astype(np.int64) * P + pos % P
    return out


@pytest.mark.parametrize("name", ["sliding_decode", "verify_block"])
def test_plan_update_in_place_matches_a_fresh_plan(name):
    """okc_attn_plan_update re-plans an existing plan for the next lengths: the
    step then equals one made with a fresh plan bit for bit; a workspace too
    small for the new plan is refused and the plan keeps its previous split."""
    import fp8_kv_paged_gb300 as okc
    from test_gpu_parity import SMALL
    cfg = W.config(name, **SMALL[name])
    inp = W.generate(cfg)
    shorter = _shorter(cfg, inp, 150)
    step = okc.AttnStep(cfg, inp["seq_lens"])
    for case in (shorter, inp, shorter):
        step.plan.update(case["seq_lens"])
        z = step.plan.sizes
        assert z == okc.okc_attn_plan_sizes(cfg, case["seq_lens"])
        assert z["o_partial_bytes"] <= step.o_partial.numel() * 4
        d = to_device(cfg, case)
        out = step.run_fused(d, eps=case["eps"])
        import torch
        torch.cuda.synchronize()
        ref = run_gpu(cfg, case, plan_form=True, fused=True)
        assert step.errors() == 0
        got = out.view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.array_equal(got, ref["out"])
        check_against_oracle(cfg, case, got, d["k_cache"].cpu().numpy(), d["v_cache"].cpu().numpy())
    # a plan whose workspace fits only short contexts refuses longer ones
    tiny = {k: (np.minimum(v, 40) if k == "seq_lens" else v) for k, v in inp.items()}
    import torch
    sz = okc.okc_attn_plan_sizes(cfg, tiny["seq_lens"])
    big = okc.okc_attn_plan_sizes(cfg, inp["seq_lens"])
    if big["workspace_bytes"] > sz["workspace_bytes"]:
        ws = torch.empty(sz["workspace_bytes"], dtype=torch.uint8, device="cuda")
        plan = okc.okc_attn_plan(cfg, tiny["seq_lens"], ws)
        with pytest.raises(okc.OkcError):
            plan.update(inp["seq_lens"])
        assert plan.sizes == sz
        plan.close()


def test_workspace_sized_for_the_longest_context_serves_every_update():
    """A workspace of okc_attn_plan_workspace_size(max context) holds the plan
    of every step up to that context: okc_attn_plan_create on short contexts,
    then okc_attn_plan_update to longer ones never runs out of room, and each
    step's sizes stay within okc_attn_plan_max_sizes (the device's own SM
    count and occupancy); okc_attn_plan_scratch_sizes equals the plan's sizes."""
    import torch
    import fp8_kv_paged_gb300 as okc
    for name in ("sliding_decode", "verify_block", "mixed_full_decode"):
        cfg = W.config(name)
        seq = W.lengths(cfg)
        max_context = int(seq.max()) + cfg["q_len"]
        nbytes = okc.okc_attn_plan_workspace_size(cfg, max_context)
        bound = okc.okc_attn_plan_max_sizes(cfg, max_context)
        assert nbytes == bound["workspace_bytes"]
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        plan = okc.okc_attn_plan_create(cfg, np.minimum(seq, 5), ws)
        rng = np.random.default_rng(5)
        for frac in (0.01, 0.3, 1.0):
            s = np.minimum(seq, (rng.random(len(seq)) * frac * max_context).astype(np.int32))
            for case in (s, seq):
                plan.update(case)
                z = plan.scratch_sizes()
                assert z == plan.sizes == okc.okc_attn_plan_sizes(cfg, case)
                for f in ("workspace_bytes", "q_fp8_bytes", "o_partial_bytes", "lse_partial_bytes", "num_work"):
                    assert z[f] <= bound[f], (name, f)
        torch.cuda.synchronize()
        plan.close()


def test_plan_update_keeps_the_device_error_word():
    """Bits the kernels set in the plan's error word survive okc_attn_plan_update
    (the update uploads the work list past the word) until
    okc_attn_plan_clear_errors zeroes it; a clean step then reports nothing."""
    import fp8_kv_paged_gb300 as okc
    import torch
    cfg = W.config("sliding_decode", batch=4, seq=("uniform", 500, 900))
    inp = W.generate(cfg)
    bad = dict(inp, page_table=inp["page_table"].copy())
    bad["page_table"][2, 10] = cfg["num_pages"] + 5  # a visible key's page past the pool
    step = okc.AttnStep(cfg, inp["seq_lens"])
    step.run_fused(to_device(cfg, bad), eps=inp["eps"])
    assert step.errors() == okc.DEVERR_PAGE
    step.plan.update(inp["seq_lens"] - 7)
    assert step.errors() == okc.DEVERR_PAGE
    okc.okc_attn_plan_clear_errors(step.plan)
    assert step.errors() == 0
    step.plan.update(inp["seq_lens"])
    out = step.run_fused(to_device(cfg, inp), eps=inp["eps"])
    torch.cuda.synchronize()
    assert step.errors() == 0
    check_against_oracle(cfg, inp, out.view(torch.int16).cpu().numpy().view(np.uint16))


def _at_lengths(cfg, inp, seq):
    """The same batch at cached lengths `seq` (each <= the batch's own): same
    caches and page table, positions, cache rows and lengths moved back."""
    out = dict(inp)
    L, P = cfg["q_len"], cfg["page_size"]
    seq = np.asarray(seq, np.int32)
    out["seq_lens"] = seq
    out["cache_seqlens"] = (seq + L).astype(np.int32)
    req = np.repeat(np.arange(cfg["batch"]), L)
    pos = seq.astype(np.int64)[req] + np.tile(np.arange(L), cfg["batch"])
    out["positions"] = pos
    out["cache_loc"] = inp["page_table"][req, pos // P].astype(np.int64) * P + pos % P
    return out


@pytest.mark.parametrize("name", ["full_decode_32k", "mixed_full_decode", "verify_block", "sliding_decode"])
def test_fixed_capacity_graph_replays_after_updates(name):
    """A fixed-capacity plan (okc_plan_options.max_context): okc_attn_step is
    captured in a CUDA graph once; then, step after step, okc_attn_plan_update
    re-plans for new lengths that change num_work, the caller rewrites the
    device inputs, and the same graph is replayed: every replay equals the
    oracle on that step's inputs (element-wise, under the acceptance bounds)."""
    import fp8_kv_paged_gb300 as okc
    import torch
    from test_gpu_parity import SMALL
    cfg = W.config(name, **SMALL[name])
    if name == "verify_block":
        cfg["window"] = 0  # (work items then grow with the context)
    inp = W.generate(cfg)
    seq = inp["seq_lens"].astype(np.int64)
    rng = np.random.default_rng(3)
    lengths = [np.minimum(seq, 40), seq, (seq * rng.uniform(0.2, 0.9, len(seq))).astype(np.int64), seq // 3, seq]
    mc = int(seq.max()) + cfg["q_len"]
    opts = {"max_context": mc}
    step = okc.AttnStep(cfg, lengths[0], opts=opts)
    d = to_device(cfg, _at_lengths(cfg, inp, lengths[0]), rope_positions=mc)  # a table for every step
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step.run_fused(d, eps=inp["eps"], stream=s)  # warm the launch path
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step.run_fused(d, eps=inp["eps"], stream=s)
    works = set()
    for sq in lengths:
        case = _at_lengths(cfg, inp, sq)
        step.plan.update(case["seq_lens"], s)
        works.add(step.plan.sizes["num_work"])
        fresh = to_device(cfg, case)
        for k in ("qkv", "positions", "cache_loc", "cache_seqlens", "cu_seqlens_q", "seq_lens", "page_table",
                  "k_cache", "v_cache"):
            d[k].copy_(fresh[k])
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert step.errors() == 0
        got = step.out.view(torch.int16).cpu().numpy().view(np.uint16)
        check_against_oracle(cfg, case, got, d["k_cache"].cpu().numpy(), d["v_cache"].cpu().numpy())
    assert len(works) > 1, works  # the updates changed the number of work items


@pytest.mark.parametrize("name", ["sliding_decode", "mixed_full_decode", "tiny_sliding_decode"])
def test_early_gather_steps_back_to_back(name):
    """OKC_PLAN_EARLY_GATHER: six one-kernel steps captured back to back in one
    CUDA graph, step i on input set i % 3 (three sets of the same lengths with
    their own qkv and caches, so no step reads what the step before it writes):
    each step overlaps its gather with its predecessor, and every output equals
    the default plan's step on the same set bit for bit, and the oracle's."""
    import fp8_kv_paged_gb300 as okc
    import torch
    from test_gpu_parity import SMALL
    cfg = W.config(name, **SMALL[name])
    inp = W.generate(cfg)
    cases = [inp]
    for k in (1, 2):
        other = W.generate(dict(cfg), seed=cfg["seed"] + 31 * k)
        cases.append(dict(inp, qkv=other["qkv"], k_cache=np.roll(inp["k_cache"], 7 * k),
                          v_cache=np.roll(inp["v_cache"], 5 * k)))
    refs = [run_gpu(cfg, c, fused=True) for c in cases]  # default plan, one kernel, eager
    flags = okc.PLAN_STEP_ONE_LAUNCH | okc.PLAN_EARLY_GATHER
    step = okc.AttnStep(cfg, inp["seq_lens"], opts={"flags": flags})
    sets = [to_device(cfg, c) for c in cases]
    outs = [torch.empty_like(step.out) for _ in range(6)]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step.run_fused(sets[0], eps=inp["eps"], stream=s)  # warm the launch path
    s.synchronize()
    sets = [to_device(cfg, c) for c in cases]  # fresh caches
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for i in range(6):
            step.run_fused(sets[i % 3], eps=inp["eps"], out=outs[i], stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert step.errors() == 0
    for i in range(6):
        got = outs[i].view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.array_equal(got, refs[i % 3]["out"]), i
    for j in range(3):
        assert np.array_equal(sets[j]["k_cache"].cpu().numpy(), refs[j]["k_cache"])
        assert np.array_equal(sets[j]["v_cache"].cpu().numpy(), refs[j]["v_cache"])
    check_against_oracle(cfg, cases[1], outs[1].view(torch.int16).cpu().numpy().view(np.uint16),
                         sets[1]["k_cache"].cpu().numpy(), sets[1]["v_cache"].cpu().numpy())
