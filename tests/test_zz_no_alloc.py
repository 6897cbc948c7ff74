"""okc_attn_decode_combine_noalloc: decode + merge + norm-gate for callers that
cannot allocate device memory (an op inside a framework that owns every device
allocation and passes the op only its inputs and outputs, or code that must not
trigger the synchronisation cudaMalloc/cudaFree can cause). Its scratch is a
static device array inside the library, so its output must equal the
three-call path's output for the same inputs, call after call, although every
call reuses (and leaves behind) the same array.

This file is collected last on purpose: a run that stops at the first failure
has run every other test before this one.
"""
import numpy as np
import pytest
import torch

import workloads as W
from parity_util import OUT_MAX_ABS, OUT_MEAN_ABS, check_against_oracle, to_device

pytestmark = pytest.mark.gpu


def _three_call(okc, cfg, inp, d):
    step = okc.AttnStep(cfg, inp["seq_lens"])
    out = step.run(d, eps=inp["eps"]).clone()
    torch.cuda.synchronize()
    assert step.errors() == 0
    return step, out


def _noalloc(okc, cfg, inp, d, q_fp8, out=None):
    if out is None:
        out = torch.full((inp["qkv"].shape[0], 16 * 64), float("nan"), dtype=torch.bfloat16, device="cuda")
    okc.okc_attn_decode_combine_noalloc(
        cfg, inp["seq_lens"], q_fp8, d["k_cache"], d["v_cache"], d["k_scale"], d["v_scale"],
        d["page_table"], d["cache_seqlens"], d["cu_seqlens_q"], d["seq_lens"], d["qkv"],
        d["norm_weight"], inp["eps"], out)
    torch.cuda.synchronize()
    return out


def _compare(out, ref):
    a = out.float().cpu().numpy()
    b = ref.float().cpu().numpy()
    assert np.all(np.isfinite(a))
    err = np.abs(a - b)
    assert err.max() <= OUT_MAX_ABS and err.mean() <= OUT_MEAN_ABS, (err.max(), err.mean())
    return float(np.mean(a == b))


def test_noalloc_matches_three_call_path(cuda_lib):
    okc = cuda_lib
    cases = [
        W.config("sliding_decode", batch=8, seq=("uniform", 1024, 3000)),
        W.config("verify_block", batch=4, seq=("uniform", 2100, 4000)),
    ]
    prepared = []
    for cfg in cases:
        inp = W.generate(cfg)
        d = to_device(cfg, inp)
        step, ref = _three_call(okc, cfg, inp, d)  # also runs okc_prepare_qkv into step.q_fp8
        prepared.append((cfg, inp, d, step, ref))
    # two calls in a row on different steps, then the first again: each one must
    # match the three-call output whatever the previous call left in the array
    for cfg, inp, d, step, ref in prepared + prepared[:1]:
        out = _noalloc(okc, cfg, inp, d, step.q_fp8)
        exact = _compare(out, ref)
        assert exact == 1.0  # same kernels, same merge order: bit-identical
        # and against the oracle on the same inputs, under the acceptance bounds
        check_against_oracle(cfg, inp, out.view(torch.int16).cpu().numpy().view(np.uint16))


def test_noalloc_call_takes_no_device_memory(cuda_lib):
    """After the first call on the device (which loads the library's module and,
    with it, the static array), further calls leave the device's free memory
    unchanged: they allocate nothing."""
    okc = cuda_lib
    cfg = W.config("sliding_decode", batch=8, seq=("uniform", 1024, 3000))
    inp = W.generate(cfg)
    d = to_device(cfg, inp)
    step, ref = _three_call(okc, cfg, inp, d)
    outs = [torch.empty_like(ref) for _ in range(3)]  # every tensor allocated up front
    _noalloc(okc, cfg, inp, d, step.q_fp8, outs[0])
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for o in outs[1:]:
        _noalloc(okc, cfg, inp, d, step.q_fp8, o)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    for o in outs:
        assert torch.equal(o, ref)


def _bad_page_step(okc, cfg, inp, d):
    """The three calls on inputs with an out-of-pool page id: they flag it."""
    step = okc.AttnStep(cfg, inp["seq_lens"])
    out = step.run(d, eps=inp["eps"]).clone()
    torch.cuda.synchronize()
    assert step.errors() == okc.DEVERR_PAGE
    return step, out


def test_noalloc_skips_a_bad_page_id(cuda_lib):
    """The entry point has no error word, so it cannot report a page id past
    the pool; its kernels still bound-check it and read nothing there. On the
    q_len 1 kernel the key reads as zeros (as in the oracle): the output equals
    the three calls' bit for bit and the oracle on every row. On the tcgen05
    kernel (verify blocks, TMA loads) the skipped rows leave that request's
    output void: every other request equals the three calls' output."""
    okc = cuda_lib
    cfg = W.config("sliding_decode", batch=4, seq=("uniform", 500, 900))
    inp = W.generate(cfg)
    inp = dict(inp, page_table=inp["page_table"].copy())
    inp["page_table"][2, 10] = cfg["num_pages"] + 5
    d = to_device(cfg, inp)
    step, ref = _bad_page_step(okc, cfg, inp, d)
    out = _noalloc(okc, cfg, inp, d, step.q_fp8)
    assert torch.equal(out, ref)
    check_against_oracle(cfg, inp, out.view(torch.int16).cpu().numpy().view(np.uint16))

    vcfg = W.config("verify_block", batch=3, seq=("list", [300, 1000, 2500]))
    vinp = W.generate(vcfg)
    vinp = dict(vinp, page_table=vinp["page_table"].copy())
    vinp["page_table"][1, 5] = vcfg["num_pages"] + 7
    vd = to_device(vcfg, vinp)
    vstep, vref = _bad_page_step(okc, vcfg, vinp, vd)
    vout = _noalloc(okc, vcfg, vinp, vd, vstep.q_fp8)
    L = vcfg["q_len"]
    for b in (0, 2):
        assert torch.equal(vout[b * L:(b + 1) * L], vref[b * L:(b + 1) * L]), b


def test_noalloc_rejects_steps_beyond_its_scratch(cuda_lib):
    okc = cuda_lib
    # 200 requests x a 16-token block: 200 work items x 256 rows of partials
    # need ~13 MB, more than the 8 MiB static array
    cfg = dict(W.config("verify_block"), batch=200, q_len=16, max_pages=4, num_pages=1000)
    dummy = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    f = torch.zeros(1 << 14, dtype=torch.float32, device="cuda")
    i32 = torch.zeros(1 << 14, dtype=torch.int32, device="cuda")
    bf = torch.zeros(1 << 15, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(okc.OkcError) as e:
        okc.okc_attn_decode_combine_noalloc(cfg, np.full(200, 100, np.int32), dummy, dummy, dummy, f, f,
                                            i32, i32, i32, i32, bf, None, 1e-5, bf)
    assert e.value.status == okc.ERR_WORKSPACE
