"""GPU parity of the one-kernel step on the tcgen05 decode (okc_attn_step under
OKC_PLAN_STEP_ONE_LAUNCH for blocks of 2..8 tokens): q and the step's new K/V
rows are derived from qkv inside the decode CTAs (the new rows put into the
tiles in place of the gathered ones and written to the cache by the CTA that
owns their keys), and the block's last CTA merges the splits and applies the
norm-gate. Against the oracle (output and written cache rows) and bit for bit
against the three-kernel step, on TMA-fed (64- and 8-row pages) and
cp.async-fed (1- and 4-row pages) tiles, with forced splits that cut the new
keys across items and put a tile's leading rows in the previous item, ragged
q lengths, scaled caches, the folded q-norm, repeated launches (the arrival
counters reset) and host-made bad inputs (flagged, nothing out of range)."""
import numpy as np
import pytest

import workloads as W
from parity_util import full_check, run_gpu, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib):
    return cuda_lib


def _one(okc, opts=None):
    return dict(opts or {}, flags=(opts or {}).get("flags", 0) | okc.PLAN_STEP_ONE_LAUNCH)


def _same_as_three_kernels(cfg, inp, opts=None):
    import fp8_kv_paged_gb300 as okc
    a = run_gpu(cfg, inp, opts)
    b = run_gpu(cfg, inp, _one(okc, opts), fused=True, plan_form=True)
    assert b["sizes"]["step_kernels"] == 1
    assert b["errors"] == 0
    assert np.array_equal(a["out"], b["out"])
    assert np.array_equal(a["k_cache"], b["k_cache"]) and np.array_equal(a["v_cache"], b["v_cache"])


CASES = [
    # q_len, page size, window, RoPE theta, kv_scale, seq range
    (8, 64, 2048, 5e5, 0.5, (2000, 5000)),   # the verify block's shape (TMA tiles)
    (8, 8, 0, 0.0, 1.0, (0, 700)),           # TMA tiles, 8-row pages, full attention
    (4, 1, 2048, 5e5, 1.0, (1500, 2600)),    # cp.async tiles
    (2, 4, 512, 5e5, 0.75, (0, 1200)),       # cp.async tiles, scaled caches
    (7, 64, 0, 5e5, 1.0, (0, 300)),          # odd block, short contexts (new keys in the first tile)
]


@pytest.mark.parametrize("L,P,window,rope,kvs,seq", CASES)
def test_one_kernel_tcgen05_step(L, P, window, rope, kvs, seq):
    cfg = W.config("verify_block", batch=6, q_len=L, page_size=P, window=window, rope_theta=rope,
                   kv_scale=kvs, seq=("uniform", *seq))
    inp = W.generate(cfg)
    full_check(cfg, inp, fused=True)  # the one-kernel form (oracle: output and caches)
    _same_as_three_kernels(cfg, inp)


@pytest.mark.parametrize("chunk", [16, 24, 60, 200])
def test_new_keys_across_items(chunk):
    """Items of 16..200 keys: the 8 new keys fall in two or three items, and a
    TMA tile starting on an 8-row boundary below its item's first key holds
    new keys of the previous item (computed by both CTAs, written by one)."""
    cfg = W.config("verify_block", batch=4, seq=("uniform", 300, 900))
    inp = W.generate(cfg)
    full_check(cfg, inp, opts={"chunk_keys": chunk}, fused=True)
    _same_as_three_kernels(cfg, inp, {"chunk_keys": chunk})


def test_ragged_q_lengths_up_to_eight():
    cfg = W.config("extend", batch=7, q_len=8, q_lens=("list", [8, 1, 0, 5, 8, 2, 3]),
                   seq=("uniform", 0, 3000), page_size=64, window=2048, rope_theta=5e5)
    inp = W.generate(cfg)
    full_check(cfg, inp, fused=True)
    _same_as_three_kernels(cfg, inp)


def test_folded_q_norm_and_distinct_scales():
    import fp8_kv_paged_gb300 as okc
    cfg = W.config("verify_block", batch=4, seq=("uniform", 1000, 3000), q_norm=okc.QNORM_FOLDED_SCALE,
                   kv_scale=0.7, k_scale=0.7, v_scale=0.6)
    inp = W.generate(cfg)
    full_check(cfg, inp, fused=True)
    _same_as_three_kernels(cfg, inp)


def test_repeated_launches_reset_the_tickets():
    import fp8_kv_paged_gb300 as okc
    import torch
    cfg = W.config("verify_block", batch=5, seq=("uniform", 2000, 4000))
    inp = W.generate(cfg)
    d = to_device(cfg, inp)
    step = okc.AttnStep(cfg, inp["seq_lens"], opts={"chunk_keys": 256, "flags": okc.PLAN_STEP_ONE_LAUNCH})
    assert step.sizes["step_kernels"] == 1
    outs = [step.run_fused(d, eps=inp["eps"]).clone() for _ in range(3)]
    torch.cuda.synchronize()
    assert step.errors() == 0
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


def test_bad_inputs_are_flagged():
    """A cache row past the pool (not written) and a position past the RoPE
    table: the one-kernel step flags each and stays in range."""
    import fp8_kv_paged_gb300 as okc
    cfg = W.config("verify_block", batch=3, seq=("uniform", 500, 900))
    inp = W.generate(cfg)
    bad = dict(inp, cache_loc=inp["cache_loc"].copy())
    bad["cache_loc"][5] = cfg["num_pages"] * cfg["page_size"] + 3
    gpu = run_gpu(cfg, bad, fused=True)
    assert gpu["sizes"]["step_kernels"] == 1
    assert gpu["errors"] & okc.DEVERR_CACHE_LOC
    d = to_device(cfg, inp, rope_positions=int(inp["positions"].max()))  # one short
    gpu = run_gpu(cfg, inp, dev_inp=d, fused=True)
    assert gpu["errors"] & okc.DEVERR_POSITION
