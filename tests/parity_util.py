"""Helpers for the GPU parity tests: upload the seeded inputs, run the block
through the C ABI, and compare with the oracle under the acceptance bounds:
  - cache rows outside cache_loc untouched, byte for byte;
  - E4M3 bytes (cache rows written, q) identical in >= 99.99% of elements and
    never more than one E4M3 step apart;
  - bf16 output: max abs error <= 2e-2 and mean abs error <= 2e-3.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads as W

FP8_MATCH_MIN = 0.9999
OUT_MAX_ABS = 2e-2
OUT_MEAN_ABS = 2e-3


def to_device(cfg: dict, inp: dict, device="cuda", rope_positions: int | None = None) -> dict:
    d = W.to_torch(inp, device)
    if cfg["rope_theta"] != 0.0:
        import fp8_kv_paged_gb300 as okc
        n = rope_positions or int(inp["positions"].max()) + 1
        d["rope_table"] = torch.empty((n, 64), dtype=torch.float32, device=device)
        okc.okc_rope_table_init(cfg["rope_theta"], n, d["rope_table"])
    return d


def run_gpu(cfg: dict, inp: dict, opts: dict | None = None, dev_inp: dict | None = None,
            fused: bool = False, plan_seq=None, plan_form: bool = False) -> dict:
    """One step through the three calls (fused=False) or okc_attn_step (fused=True:
    in its one-kernel form wherever that exists, or in the form the plan chooses
    with plan_form=True). plan_seq: host lengths the plan is made with (default:
    the inputs' own)."""
    import fp8_kv_paged_gb300 as okc
    d = dev_inp if dev_inp is not None else to_device(cfg, inp)
    if fused and not plan_form:
        opts = dict(opts or {}, flags=(opts or {}).get("flags", 0) | okc.PLAN_STEP_ONE_LAUNCH)
    step = okc.AttnStep(cfg, inp["seq_lens"] if plan_seq is None else plan_seq, opts=opts,
                        q_lens=inp["q_lens"] if "q_lens" in cfg else None)
    out = step.run_fused(d, eps=inp["eps"]) if fused else step.run(d, eps=inp["eps"])
    torch.cuda.synchronize()
    T = inp["qkv"].shape[0]
    return {
        "out": out.view(torch.int16).cpu().numpy().view(np.uint16),
        "k_cache": d["k_cache"].cpu().numpy(),
        "v_cache": d["v_cache"].cpu().numpy(),
        "q8": step.q_fp8[: T * 16 * 64].cpu().numpy().reshape(T, 16, 64),
        "errors": step.errors(),
        "sizes": step.sizes,
        "step": step,
    }


def e4m3_ulps(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in E4M3 steps (codes are monotone in magnitude for each sign)."""
    def ordinal(c):
        c = c.astype(np.int32)
        return np.where(c >= 0x80, -(c & 0x7F), c)
    return np.abs(ordinal(a) - ordinal(b))


def check_fp8(gpu: np.ndarray, ref: np.ndarray, what: str) -> dict:
    eq = np.mean(gpu == ref) if gpu.size else 1.0
    ulps = int(e4m3_ulps(gpu, ref).max()) if gpu.size else 0
    assert eq >= FP8_MATCH_MIN, f"{what}: only {eq:.6f} of E4M3 bytes identical"
    assert ulps <= 1, f"{what}: E4M3 bytes {ulps} steps apart"
    return {"match": float(eq), "max_ulps": ulps}


def check_caches(inp: dict, gpu: dict, ref_k: np.ndarray, ref_v: np.ndarray) -> dict:
    loc = inp["cache_loc"]
    rows = ref_k.reshape(-1, 128).shape[0]
    touched = np.zeros(rows, bool)
    valid = (loc >= 0) & (loc < rows)
    touched[loc[valid]] = True
    res = {}
    for name, g, r, orig in (("k_cache", gpu["k_cache"], ref_k, inp["k_cache"]),
                             ("v_cache", gpu["v_cache"], ref_v, inp["v_cache"])):
        g2, r2, o2 = g.reshape(rows, 128), r.reshape(rows, 128), orig.reshape(rows, 128)
        assert np.array_equal(g2[~touched], o2[~touched]), f"{name}: rows outside cache_loc changed"
        res[name] = check_fp8(g2[touched], r2[touched], name)
    return res


def check_out(gpu_bits: np.ndarray, ref_bits: np.ndarray, rows_mask: np.ndarray | None = None) -> dict:
    g = oracle.bf16_value(gpu_bits).reshape(ref_bits.shape[0], 16, 64)
    r = oracle.bf16_value(ref_bits).reshape(ref_bits.shape[0], 16, 64)
    if rows_mask is not None:
        g, r = g[rows_mask.astype(bool)], r[rows_mask.astype(bool)]
    assert np.all(np.isfinite(g)), "non-finite output"
    err = np.abs(g - r)
    mx, mean = float(err.max()), float(err.mean())
    assert mx <= OUT_MAX_ABS, f"max abs error {mx}"
    assert mean <= OUT_MEAN_ABS, f"mean abs error {mean}"
    return {"max_abs": mx, "mean_abs": mean, "exact": float(np.mean(g == r))}


def oracle_ref(cfg: dict, inp: dict, rows_mask=None) -> dict:
    """The oracle's step on copies of the caches: q8, caches, bf16 out bits."""
    return oracle.step(cfg, inp, rows_mask)


def check_against_oracle(cfg: dict, inp: dict, out_bits: np.ndarray, k_cache=None, v_cache=None,
                         ref: dict | None = None) -> dict:
    """A step's output (bf16 bits [T, Hq*64]) and, when given, its caches after
    the step, against the oracle on the same inputs under the acceptance bounds."""
    ref = ref if ref is not None else oracle_ref(cfg, inp)
    rep = {"out": check_out(np.asarray(out_bits).reshape(ref["out"].shape), ref["out"])}
    if k_cache is not None:
        rep.update(check_caches(inp, {"k_cache": k_cache, "v_cache": v_cache}, ref["k_cache"], ref["v_cache"]))
    return rep


def full_check(cfg: dict, inp: dict, opts: dict | None = None, rows_mask=None, expect_errors: int = 0,
               fused: bool = False, plan_seq=None, plan_form: bool = False):
    gpu = run_gpu(cfg, inp, opts, fused=fused, plan_seq=plan_seq, plan_form=plan_form)
    k = inp["k_cache"].copy()
    v = inp["v_cache"].copy()
    q8, _ = oracle.prepare(cfg, inp, k, v)
    rep = {} if fused else {"q8": check_fp8(gpu["q8"], q8, "q8")}
    rep.update(check_caches(inp, gpu, k, v))
    o, _ = oracle.attention(cfg, inp, q8, k, v, rows_mask)
    ref = oracle.normgate(cfg, o, inp["qkv"], inp.get("norm_weight"), inp["eps"], rows_mask)
    rep["out"] = check_out(gpu["out"], ref, rows_mask)
    assert gpu["errors"] == expect_errors, f"device error word {gpu['errors']:#x}"
    rep["num_work"] = gpu["sizes"]["num_work"]
    rep["step_kernels"] = gpu["sizes"]["step_kernels"]
    return rep
