"""GPU parity of prefill / extend steps: per-request q lengths (the problem
file's ragged cu_seqlens_q with its max_seqlen_q) on the same paged FP8 cache.
Batches mix decode requests (1 token), extends of 37, 256 and 1024 tokens and
requests with no new token, at window 2048 and 0, on 1-, 16- and 64-row pages;
through the three calls (the tcgen05 decode on blocks of 16 tokens, one softmax
warpgroup per KV head), through
okc_attn_step, on the warp-level kernel (blocks of 16 tokens) and with forced
split sizes; against the oracle on sampled query rows (every request's first
and last token always in the sample). Uniform q lengths past 8 (several query
blocks per request), in-place varlen plan updates and the extend workload at
full size follow."""
import numpy as np
import pytest
import torch

import workloads as W
from parity_util import check_against_oracle, full_check, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib):
    return cuda_lib


def _rows_mask(inp, frac, seed=0):
    """A uniform sample of the (token, head) rows plus every head of each
    request's first and last new token."""
    T = inp["qkv"].shape[0]
    rng = np.random.default_rng(seed)
    m = (rng.random((T, 16)) < frac).astype(np.uint8)
    cu = inp["cu_seqlens_q"]
    for b in range(len(cu) - 1):
        if cu[b + 1] > cu[b]:
            m[cu[b]] = 1
            m[cu[b + 1] - 1] = 1
    return m


def _extend_cfg(q_lens, seq, window, P, rope, kv_scale=1.0):
    return W.config("extend", batch=len(q_lens), q_len=max(q_lens), q_lens=("list", list(q_lens)),
                    seq=("uniform", *seq), window=window, page_size=P, rope_theta=rope, kv_scale=kv_scale)


CASES = [
    # q lengths, seq_lens range, window, page size, RoPE theta, kv_scale
    ([1, 37, 256, 1024, 0, 5], (0, 3000), 2048, 64, 5e5, 1.0),
    ([1, 37, 256, 1024, 0, 5], (0, 3000), 0, 64, 0.0, 1.0),
    ([1024, 1, 37], (2040, 2100), 2048, 1, 5e5, 0.5),
    ([256, 256, 9, 16, 17, 1], (0, 500), 0, 16, 0.0, 1.0),
]


@pytest.mark.parametrize("q_lens,seq,window,P,rope,kvs", CASES)
def test_ragged_extend_batches(q_lens, seq, window, P, rope, kvs):
    import fp8_kv_paged_gb300 as okc
    cfg = _extend_cfg(q_lens, seq, window, P, rope, kvs)
    inp = W.generate(cfg)
    mask = _rows_mask(inp, 0.2, seed=len(q_lens))
    rep = full_check(cfg, inp, rows_mask=mask)  # three calls, tcgen05 decode, blocks of 16
    assert rep["q8"]["match"] == 1.0
    full_check(cfg, inp, rows_mask=mask, fused=True, plan_form=True)  # okc_attn_step
    full_check(cfg, inp, rows_mask=mask, opts={"flags": okc.PLAN_NO_TCGEN05})  # warp-level MMA, blocks of 16
    full_check(cfg, inp, rows_mask=mask, opts={"chunk_keys": 200})  # several splits per block


@pytest.mark.parametrize("L,P,window", [(12, 64, 2048), (40, 1, 0), (16, 8, 0)])
def test_uniform_q_len_past_one_block(L, P, window):
    """A uniform q_len of more than 8 tokens: every request is several query
    blocks (tcgen05) or one or more of 16 (warp-level kernel)."""
    import fp8_kv_paged_gb300 as okc
    cfg = W.config("verify_block", batch=5, q_len=L, page_size=P, window=window, seq=("uniform", 100, 3000))
    inp = W.generate(cfg)
    full_check(cfg, inp)
    full_check(cfg, inp, fused=True, plan_form=True)
    full_check(cfg, inp, opts={"flags": okc.PLAN_NO_TCGEN05})


def test_varlen_plan_update_in_place():
    """okc_attn_plan_update_varlen re-plans a varlen plan for new q lengths
    (same workspace, sized by okc_attn_plan_max_sizes): each step equals the
    oracle on its own inputs."""
    import fp8_kv_paged_gb300 as okc
    base = _extend_cfg([1, 37, 256, 1024, 5], (0, 2000), 0, 64, 0.0)
    steps = [[1, 37, 256, 1024, 5], [3, 0, 1, 64, 200], [1024, 1024, 1, 1, 1]]
    cfgs, inps = [], []
    for i, ql in enumerate(steps):
        c = dict(base, q_lens=("list", ql), seed=500 + i)
        cfgs.append(c)
        inps.append(W.generate(c))
    mc = max(int((x["seq_lens"] + x["q_lens"]).max()) for x in inps)
    # one config for every step: the largest page table and pool (smaller pools
    # padded with pages no request uses)
    NP, MP = max(c["num_pages"] for c in cfgs), max(c["max_pages"] for c in cfgs)
    for c, inp in zip(cfgs, inps):
        for k in ("k_cache", "v_cache"):
            pad = np.zeros((NP - c["num_pages"],) + inp[k].shape[1:], np.uint8)
            inp[k] = np.concatenate([inp[k], pad])
        c["num_pages"], c["max_pages"] = NP, MP
    bound = okc.okc_attn_plan_max_sizes(cfgs[0], mc)
    ws = torch.empty(bound["workspace_bytes"], dtype=torch.uint8, device="cuda")
    q8 = torch.empty(bound["q_fp8_bytes"], dtype=torch.uint8, device="cuda")
    op = torch.empty(bound["o_partial_bytes"] // 4, dtype=torch.float32, device="cuda")
    lp = torch.empty(bound["lse_partial_bytes"] // 4, dtype=torch.float32, device="cuda")
    plan = okc.okc_attn_plan(cfgs[0], inps[0]["seq_lens"], ws, q_lens=inps[0]["q_lens"])
    for i, (c, inp) in enumerate(zip(cfgs, inps)):
        pt = np.full((c["batch"], c["max_pages"]), -1, np.int32)
        pt[:, :inp["page_table"].shape[1]] = inp["page_table"]
        inp = dict(inp, page_table=pt)
        if i:
            plan.update(inp["seq_lens"], q_lens=inp["q_lens"])
        assert plan.sizes == okc.okc_attn_plan_sizes(c, inp["seq_lens"], q_lens=inp["q_lens"])
        d = to_device(c, inp)
        T = inp["qkv"].shape[0]
        out = torch.empty((T, 1024), dtype=torch.bfloat16, device="cuda")
        okc.okc_prepare_qkv(plan, d["qkv"], d["positions"], d["cache_loc"], d["k_cache"], d["v_cache"],
                            d["k_scale"], d["v_scale"], d["rope_table"], q8)
        okc.okc_attn_decode(plan, q8, d["k_cache"], d["v_cache"], d["k_scale"], d["v_scale"], d["page_table"],
                            d["cache_seqlens"], d["cu_seqlens_q"], d["seq_lens"], op, lp)
        okc.okc_attn_combine_normgate(plan, op, lp, d["qkv"], d["norm_weight"], inp["eps"], out)
        torch.cuda.synchronize()
        assert okc.okc_attn_plan_read_errors(plan) == 0
        mask = _rows_mask(inp, 0.2, seed=i)
        ref = __import__("oracle").step(c, inp, mask)
        from parity_util import check_out
        check_out(out.view(torch.int16).cpu().numpy().view(np.uint16), ref["out"], mask)
    plan.close()


def test_q_lengths_that_disagree_with_the_plan_are_flagged():
    """Device cu_seqlens_q that differ from the plan's q lengths: the kernels
    flag OKC_DEVERR_LENGTHS (the step's output is void) and stay in bounds."""
    import fp8_kv_paged_gb300 as okc
    from parity_util import run_gpu
    cfg = _extend_cfg([37, 256, 8], (100, 900), 0, 16, 0.0)
    inp = W.generate(cfg)
    d = to_device(cfg, inp)
    cu = inp["cu_seqlens_q"].copy()
    cu[1] += 3  # request 0 now claims 40 tokens, request 1 253
    d["cu_seqlens_q"] = torch.from_numpy(cu).cuda()
    gpu = run_gpu(cfg, inp, dev_inp=d)
    assert gpu["errors"] & okc.DEVERR_LENGTHS


def test_extend_workload_full_size():
    """The benchmark's extend workload (16 requests, q lengths from {1, 37, 256,
    1024}, seq_lens up to 16384, full attention, 64-row pages) in the launch
    form the benchmark times, on a 1 % row sample plus every request's first and
    last token."""
    cfg = W.config("extend")
    inp = W.generate(cfg)
    mask = _rows_mask(inp, 0.01, seed=7)
    rep = full_check(cfg, inp, rows_mask=mask, fused=True, plan_form=True)
    print("extend", rep)
