"""The RMS inverse of steps 1-3 is the float32 rounding of the exact
1/sqrt(sum(x^2)/64 + eps) (the oracle's reading). The kernels compute it in
float32 with a double-precision fallback next to rounding boundaries; this
stress test feeds heads chosen to reach every branch: per-head scales across
2^-60..2^60, per-element exponent spreads, all-zero heads, and values whose
squares overflow float32 (fallback). q and the written cache rows must match
the oracle byte for byte, through okc_prepare_qkv and through okc_attn_step."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from parity_util import run_gpu

pytestmark = pytest.mark.gpu

HQ, HKV, D = 16, 2, 64


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib):
    return cuda_lib


def _adversarial_qkv(T, rng):
    width = (2 * HQ + 2 * HKV) * D
    x = rng.standard_normal((T, width)).astype(np.float64)
    heads = x[:, : (HQ + 2 * HKV) * D].reshape(T, HQ + 2 * HKV, D)
    kind = rng.integers(0, 6, size=(T, HQ + 2 * HKV))
    scale = np.exp2(rng.integers(-60, 61, size=(T, HQ + 2 * HKV)))[..., None]
    spread = np.exp2(rng.integers(-40, 41, size=heads.shape))
    heads = np.where((kind == 1)[..., None], heads * scale, heads)
    heads = np.where((kind == 2)[..., None], heads * spread, heads)
    heads = np.where((kind == 3)[..., None], 0.0, heads)
    heads = np.where((kind == 4)[..., None], heads * 3e20, heads)        # squares overflow float32
    heads = np.where((kind == 5)[..., None], np.round(heads * 4) / 4, heads)  # few distinct values
    x[:, : (HQ + 2 * HKV) * D] = heads.reshape(T, -1)
    return oracle.bf16_bits(np.clip(x, -3e38, 3e38))


@pytest.mark.parametrize("rope,fused,L", [(0.0, False, 1), (5e5, False, 1), (5e5, True, 1), (5e5, True, 8)])
def test_rms_inverse_exact_on_adversarial_heads(rope, fused, L):
    """(L = 8 with fused: the one-kernel tcgen05 step, whose q rows are derived one
    per thread inside the decode: its output equals the three calls' bit for bit,
    whose q bytes equal the oracle's.)"""
    if L == 1:
        cfg = W.config("sliding_decode", batch=2048, seq=("uniform", 0, 40), rope_theta=rope, window=0)
    else:
        cfg = W.config("verify_block", batch=256, q_len=L, seq=("uniform", 0, 40), rope_theta=rope, window=0,
                       kv_scale=1.0)
    inp = W.generate(cfg)
    inp["qkv"] = _adversarial_qkv(inp["qkv"].shape[0], np.random.default_rng(77))
    gpu = run_gpu(cfg, inp, fused=fused)
    k = inp["k_cache"].copy()
    v = inp["v_cache"].copy()
    q8, _ = oracle.prepare(cfg, inp, k, v)
    loc = inp["cache_loc"]
    if not fused:
        assert np.array_equal(gpu["q8"], q8)
    elif L > 1:
        three = run_gpu(cfg, inp)
        assert np.array_equal(three["q8"], q8)
        assert gpu["sizes"]["step_kernels"] == 1
        assert np.array_equal(gpu["out"], three["out"])
    assert np.array_equal(gpu["k_cache"].reshape(-1, 128)[loc], k.reshape(-1, 128)[loc])
    assert np.array_equal(gpu["v_cache"].reshape(-1, 128)[loc], v.reshape(-1, 128)[loc])
