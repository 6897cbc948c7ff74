"""GPU parity: the CUDA path through the C ABI against the oracle, on seeded
inputs of the five workloads' shapes at sizes the oracle finishes in seconds
(several tiles, ragged tails), plus edge cases and forced split counts."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from parity_util import full_check, run_gpu, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib):
    return cuda_lib


SMALL = {
    "tiny_sliding_decode": {},
    "sliding_decode": dict(batch=8, seq=("uniform", 1024, 3000)),
    "full_decode_32k": dict(batch=4, seq=("const", 5000)),
    "verify_block": dict(batch=4, seq=("uniform", 2100, 4000)),
    "mixed_full_decode": dict(batch=16, seq=("loguniform", 1, 20000)),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_workload_shapes_small(name):
    cfg = W.config(name, **SMALL[name])
    inp = W.generate(cfg)
    rep = full_check(cfg, inp)
    print(name, rep)


@pytest.mark.parametrize("chunk", [16, 64, 100, 448, 100000])
@pytest.mark.parametrize("name", ["sliding_decode", "verify_block"])
def test_forced_split_sizes(name, chunk):
    cfg = W.config(name, **SMALL[name])
    inp = W.generate(cfg)
    full_check(cfg, inp, opts={"chunk_keys": chunk})


@pytest.mark.parametrize("seq,L,window,P", [
    ([0, 1, 2, 3], 1, 2048, 1),             # empty history (padded slots)
    ([0, 5, 70, 129], 8, 2048, 64),         # verify block from position 0
    ([2046, 2047, 2048, 2049], 1, 2048, 1),  # window edge
    ([2040, 2041, 2047, 2055], 8, 2048, 1),  # window edge inside the block
    ([4097], 1, 0, 1),                       # B = 1
    ([300, 17, 1000], 2, 0, 4),
    ([300, 17, 1000], 4, 256, 16),
    ([900, 33], 16, 512, 256),
    ([63, 64, 65, 127, 128, 129], 1, 64, 64),
    ([0, 5, 3000], 1, 1, 1),                 # window 1: each query sees only its own key
    ([0, 5, 3000], 8, 1, 16),
])
def test_edge_shapes(seq, L, window, P):
    cfg = W.config("tiny_sliding_decode", batch=len(seq), q_len=L, window=window, page_size=P,
                   seq=("list", seq))
    inp = W.generate(cfg)
    full_check(cfg, inp)
    full_check(cfg, inp, opts={"chunk_keys": 32})


def test_norm_weight_none_and_no_rope_scaled():
    cfg = W.config("verify_block", batch=3, seq=("uniform", 100, 900), norm_weight=False,
                   rope_theta=0.0, kv_scale=0.75)
    inp = W.generate(cfg)
    assert inp["norm_weight"] is None
    full_check(cfg, inp)


@pytest.mark.parametrize("name", ["verify_block", "sliding_decode"])
def test_distinct_k_and_v_scales(name):
    """The scaled cache path with k_scale != v_scale, both non-dyadic (0.7 and
    0.6: the bf16 cast after the division changes E4M3 codes), through the three
    calls and through okc_attn_step in both of its forms."""
    cfg = W.config(name, **SMALL[name], kv_scale=0.7, k_scale=0.7, v_scale=0.6)
    inp = W.generate(cfg)
    assert inp["k_scale"] != inp["v_scale"]
    full_check(cfg, inp)
    full_check(cfg, inp, fused=True)
    full_check(cfg, inp, fused=True, plan_form=True)


@pytest.mark.parametrize("name", ["sliding_decode", "verify_block", "full_decode_32k", "tiny_sliding_decode"])
def test_folded_q_norm(name):
    """q_norm = OKC_QNORM_FOLDED_SCALE (the vLLM qk_norm with the query factor as
    its output scale): q bytes bit-identical to the oracle's mode, the softmax
    scale sm_scale alone; through the three calls and okc_attn_step."""
    import fp8_kv_paged_gb300 as okc
    cfg = W.config(name, **SMALL[name], q_norm=okc.QNORM_FOLDED_SCALE)
    inp = W.generate(cfg)
    rep = full_check(cfg, inp)
    assert rep["q8"]["match"] == 1.0
    full_check(cfg, inp, fused=True)
    full_check(cfg, inp, fused=True, plan_form=True)


def test_rope_table_matches_oracle_rows():
    import fp8_kv_paged_gb300 as okc
    n = 140000
    tab = torch.empty((n, 64), dtype=torch.float32, device="cuda")
    okc.okc_rope_table_init(5e5, n, tab)
    host = tab.cpu().numpy()
    rng = np.random.default_rng(2)
    for pos in list(rng.integers(0, n, 200)) + [0, 1, n - 1]:
        c, s = oracle.rope_row(5e5, int(pos))
        assert np.array_equal(host[pos, :32], c) and np.array_equal(host[pos, 32:], s), pos


def test_bad_inputs_flag_errors_without_faulting():
    """Host-made bad inputs that the kernels bound-check: an out-of-pool page id,
    an out-of-pool cache row, a position past the RoPE table, inconsistent
    lengths. Each sets its error bit; nothing is read or written out of range."""
    import fp8_kv_paged_gb300 as okc
    cfg = W.config("sliding_decode", batch=4, seq=("uniform", 500, 900))
    inp = W.generate(cfg)
    # 1) a page id past the pool for a visible key of request 2: read as zeros
    bad = dict(inp, page_table=inp["page_table"].copy())
    bad["page_table"][2, 10] = cfg["num_pages"] + 5
    full_check(cfg, bad, expect_errors=okc.DEVERR_PAGE)
    # 2) a cache row past the pool: not written
    bad = dict(inp, cache_loc=inp["cache_loc"].copy())
    bad["cache_loc"][1] = cfg["num_pages"] * cfg["page_size"] + 3
    gpu = run_gpu(cfg, bad)
    assert gpu["errors"] & okc.DEVERR_CACHE_LOC
    # 3) a position past the RoPE table
    d = to_device(cfg, inp, rope_positions=int(inp["positions"].max()))  # one short
    gpu = run_gpu(cfg, inp, dev_inp=d)
    assert gpu["errors"] & okc.DEVERR_POSITION
    # 4) device seq_lens inconsistent with cache_seqlens (the plan keeps the true ones)
    d = to_device(cfg, dict(inp, seq_lens=inp["seq_lens"] + 1))
    gpu = run_gpu(cfg, inp, dev_inp=d)
    assert gpu["errors"] & okc.DEVERR_LENGTHS
    # 5) a page id past the pool in a verify block on 64-row pages (the TMA
    # loads of the tcgen05 decode skip it)
    vcfg = W.config("verify_block", batch=3, seq=("list", [300, 1000, 2500]))
    vinp = W.generate(vcfg)
    vbad = dict(vinp, page_table=vinp["page_table"].copy())
    vbad["page_table"][1, 5] = vcfg["num_pages"] + 7
    gpu = run_gpu(vcfg, vbad)
    assert gpu["errors"] & okc.DEVERR_PAGE


@pytest.mark.parametrize("fused", [False, True])
def test_plan_lengths_longer_than_device_lengths(fused):
    """A plan made for longer requests than the step's device lengths still
    covers every key: the kernels start from the plan's key ranges, find that
    the device lengths differ, reload the page ids and follow the device
    lengths (results equal the oracle's on the device lengths)."""
    cfg = W.config("sliding_decode", batch=6, seq=("uniform", 500, 3000))
    inp = W.generate(cfg)
    pad = np.full((cfg["batch"], 64), -1, np.int32)  # room in the page table for the plan's lengths
    inp["page_table"] = np.concatenate([inp["page_table"], pad], axis=1)
    cfg["max_pages"] += 64
    plan_seq = inp["seq_lens"] + 37
    full_check(cfg, inp, plan_seq=plan_seq, fused=fused)
    full_check(cfg, inp, opts={"chunk_keys": 96}, plan_seq=plan_seq, fused=fused)


def test_plan_lengths_longer_than_device_lengths_verify_block():
    """The same for a verify block on 64-row pages: the tcgen05 decode's TMA
    tiles start from the device lengths' key ranges (rounded down to 8)."""
    cfg = W.config("verify_block", batch=5, seq=("uniform", 300, 3000))
    inp = W.generate(cfg)
    pad = np.full((cfg["batch"], 2), -1, np.int32)  # room in the page table for the plan's lengths
    inp["page_table"] = np.concatenate([inp["page_table"], pad], axis=1)
    cfg["max_pages"] += 2
    plan_seq = inp["seq_lens"] + 45
    full_check(cfg, inp, plan_seq=plan_seq)
    full_check(cfg, inp, opts={"chunk_keys": 200}, plan_seq=plan_seq)


@pytest.mark.parametrize("seq,L,P,kv_scale", [
    ([100, 300], 8, 64, 0.5),
    ([2100, 2600, 4000, 70], 8, 64, 0.5),
    ([50, 900, 2047, 2048, 2049], 2, 1, 1.0),
    ([0, 1, 63, 64, 65], 4, 16, 1.0),
    ([5000, 3], 6, 64, 0.5),
    ([31, 500, 1999, 7], 3, 8, 1.0),         # pages of one 8-row TMA box
    ([1000, 4100, 2053], 8, 32, 0.5),
])
def test_verify_block_both_decode_kernels(seq, L, P, kv_scale):
    """Blocks of 2..8 tokens decode on the tcgen05 kernel by default and on the
    warp-level MMA kernel with OKC_PLAN_NO_TCGEN05: both within the bounds
    against the oracle, with forced split sizes too."""
    import fp8_kv_paged_gb300 as okc
    cfg = W.config("verify_block", batch=len(seq), q_len=L, page_size=P, kv_scale=kv_scale, seq=("list", seq))
    inp = W.generate(cfg)
    for flags in (0, okc.PLAN_NO_TCGEN05):
        full_check(cfg, inp, opts={"flags": flags} if flags else None)
        full_check(cfg, inp, opts={"flags": flags, "chunk_keys": 100})


def test_empty_batch_is_a_no_op():
    """B = 0: the plan is valid and every call returns OK without launching."""
    import fp8_kv_paged_gb300 as okc
    cfg = dict(W.config("sliding_decode"), batch=0, max_pages=1, num_pages=1)
    seq = np.zeros(0, np.int32)
    sizes = okc.okc_attn_plan_sizes(cfg, seq)
    assert sizes["num_work"] == 0 and sizes["num_tokens"] == 0
    step = okc.AttnStep(cfg, seq)
    z8 = torch.zeros(16, dtype=torch.uint8, device="cuda")
    zf = torch.zeros(16, dtype=torch.float32, device="cuda")
    zi = torch.zeros(16, dtype=torch.int32, device="cuda")
    zl = torch.zeros(16, dtype=torch.int64, device="cuda")
    zb = torch.zeros((1, 2304), dtype=torch.bfloat16, device="cuda")
    d = {"qkv": zb, "positions": zl, "cache_loc": zl, "k_cache": z8, "v_cache": z8, "k_scale": zf,
         "v_scale": zf, "page_table": zi, "cache_seqlens": zi, "cu_seqlens_q": zi, "seq_lens": zi,
         "norm_weight": None, "rope_table": torch.zeros((4, 64), dtype=torch.float32, device="cuda")}
    step.run(d)
    step.run_fused(d)
    torch.cuda.synchronize()
    assert step.errors() == 0


@pytest.mark.parametrize("L", [1, 4])
def test_many_requests(L):
    """1500 short requests: many more work items than resident CTA slots."""
    cfg = W.config("sliding_decode", batch=1500, q_len=L, seq=("uniform", 0, 400))
    inp = W.generate(cfg)
    rep = full_check(cfg, inp)
    assert rep["num_work"] >= 1500
    full_check(cfg, inp, fused=True, plan_form=True)
    full_check(cfg, inp, fused=True)


def test_forced_occupancy_plans_launch_in_a_fresh_process():
    """A plan made with okc_plan_options.ctas_per_sm / sm_count (which skip the
    occupancy query) still launches: the plan raises the decode kernels'
    shared-memory limits itself. Run in a fresh process, where no earlier plan
    has raised them, for the q_len-1 and the tcgen05 kernels."""
    import os
    import subprocess
    import sys
    code = r"""
import sys
sys.path.insert(0, "tests"); sys.path.insert(0, ".")
import workloads as W
from parity_util import full_check
for name in ("sliding_decode", "verify_block"):
    from test_gpu_parity import SMALL
    cfg = W.config(name, **SMALL[name])
    inp = W.generate(cfg)
    full_check(cfg, inp, opts={"ctas_per_sm": 1, "sm_count": 148})
print("ok")
"""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-2000:]
