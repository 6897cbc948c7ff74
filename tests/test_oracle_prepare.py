"""Pins of the oracle's steps 1-3 (`_prepare_qkv` of the Muse Spark attention
problem file "012-attention-local-splits.py"): where rows land, which columns
feed which head, RoPE as a rotation, RMS normalisation, and the scaled path —
each checked by an invariant or an independent formulation, not by re-running
the oracle's own formula.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W

HQ, HKV, D = 16, 2, 64
QCOL, KCOL, VCOL, GCOL = 0, HQ * D, (HQ + HKV) * D, (HQ + 2 * HKV) * D


def _small(**kw):
    cfg = W.config("tiny_sliding_decode", **kw)
    inp = W.generate(cfg)
    return cfg, inp


def _run(cfg, inp):
    k = inp["k_cache"].copy()
    v = inp["v_cache"].copy()
    q8, skipped = oracle.prepare(cfg, inp, k, v)
    return q8, k, v, skipped


def _torch_e4m3(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_golden_layout_facts():
    """The page's stated layout (tests/golden/page_facts.json) is what the
    generator produces."""
    import json, os
    facts = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_facts.json")))
    cfg, inp = _small()
    assert inp["qkv"].shape[1] == facts["qkv_width"]["value"]
    assert [QCOL, KCOL, VCOL, GCOL] == facts["qkv_column_starts"]["value"]
    assert cfg["eps"] == facts["rms_eps"]["value"]
    assert W.ROPE_POSITIONS == facts["rope_positions"]["value"]
    assert np.array_equal(inp["cache_seqlens"], inp["seq_lens"] + cfg["q_len"])


def test_rows_land_exactly_at_cache_loc():
    cfg, inp = _small()
    q8, k, v, skipped = _run(cfg, inp)
    assert skipped == 0
    rows_k = k.reshape(-1, HKV * D)
    rows_v = v.reshape(-1, HKV * D)
    old_k = inp["k_cache"].reshape(-1, HKV * D)
    old_v = inp["v_cache"].reshape(-1, HKV * D)
    touched = np.zeros(rows_k.shape[0], bool)
    touched[inp["cache_loc"]] = True
    assert np.array_equal(rows_k[~touched], old_k[~touched])
    assert np.array_equal(rows_v[~touched], old_v[~touched])
    # cache_loc is the page table's row of position seq_len + i
    P = cfg["page_size"]
    for t, pos in enumerate(inp["positions"]):
        b = t // cfg["q_len"]
        assert inp["cache_loc"][t] == inp["page_table"][b, pos // P] * P + pos % P
    # unscaled V is the E4M3 cast of the raw v columns (torch's cast as reference)
    for t, slot in enumerate(inp["cache_loc"]):
        raw = oracle.bf16_value(inp["qkv"][t, VCOL:VCOL + HKV * D])
        assert np.array_equal(rows_v[slot], _torch_e4m3(raw))


def test_out_of_pool_rows_are_skipped():
    cfg, inp = _small()
    inp["cache_loc"] = inp["cache_loc"].copy()
    inp["cache_loc"][0] = cfg["num_pages"] * cfg["page_size"]  # one past the pool
    q8, k, v, skipped = _run(cfg, inp)
    assert skipped == 1


@pytest.mark.parametrize("which,cols,check", [
    ("gate", (GCOL, GCOL + HQ * D), "none"),
    ("q3", (QCOL + 3 * D, QCOL + 4 * D), "q3"),
    ("k1", (KCOL + D, KCOL + 2 * D), "k1"),
    ("v0", (VCOL, VCOL + D), "v0"),
])
def test_columns_feed_only_their_head(which, cols, check):
    cfg, inp = _small()
    q8a, ka, va, _ = _run(cfg, inp)
    inp2 = dict(inp)
    qkv = inp["qkv"].copy()
    rng = np.random.default_rng(5)
    qkv[:, cols[0]:cols[1]] = W._bf16_bits(rng.standard_normal((qkv.shape[0], cols[1] - cols[0])))
    inp2["qkv"] = qkv
    q8b, kb, vb, _ = _run(cfg, inp2)
    loc = inp["cache_loc"]
    dq = np.any(q8a != q8b, axis=2)                     # [T, Hq]
    dk = np.any(ka.reshape(-1, HKV, D)[loc] != kb.reshape(-1, HKV, D)[loc], axis=2)
    dv = np.any(va.reshape(-1, HKV, D)[loc] != vb.reshape(-1, HKV, D)[loc], axis=2)
    exp_q = np.zeros_like(dq); exp_k = np.zeros_like(dk); exp_v = np.zeros_like(dv)
    if check == "q3":
        exp_q[:, 3] = True
    if check == "k1":
        exp_k[:, 1] = True
    if check == "v0":
        exp_v[:, 0] = True
    assert np.array_equal(dq, exp_q) and np.array_equal(dk, exp_k) and np.array_equal(dv, exp_v)


def test_rope_at_position_zero_is_identity():
    cfg, inp = _small()
    inp = dict(inp, positions=np.zeros_like(inp["positions"]))
    q_rope, k_rope, _, _ = _run(cfg, inp)
    q_plain, k_plain, _, _ = _run(dict(cfg, rope_theta=0.0), inp)
    assert np.array_equal(q_rope, q_plain)
    assert np.array_equal(k_rope, k_plain)


def test_rope_is_the_complex_rotation():
    """(y_2i + i*y_2i+1) * exp(i * pos * theta^(-2i/64)): the dequantised q/k
    agree with the rotation of the normalised head within E4M3 + bf16 rounding.
    Catches a swapped sign, a wrong partner or a wrong frequency index."""
    cfg, inp = _small()
    rng = np.random.default_rng(3)
    pos = rng.integers(1, 100000, size=inp["positions"].shape)
    inp = dict(inp, positions=pos)
    q8, k, _, _ = _run(cfg, inp)
    deq_q = oracle.e4m3_value(q8)
    deq_k = oracle.e4m3_value(k.reshape(-1, HKV, D)[inp["cache_loc"]])
    inv = np.float64(5e5) ** (-np.arange(0, D, 2) / D)
    worst = 0.0
    for t in range(q8.shape[0]):
        x = oracle.bf16_value(inp["qkv"][t, : (HQ + HKV) * D]).reshape(HQ + HKV, D)
        y = x / np.sqrt((x * x).mean(axis=1, keepdims=True) + 1e-5)
        z = (y[:, 0::2] + 1j * y[:, 1::2]) * np.exp(1j * pos[t] * inv)[None, :]
        rot = np.empty_like(y)
        rot[:, 0::2], rot[:, 1::2] = z.real, z.imag
        mag = np.repeat(np.abs(z), 2, axis=1)
        got = np.concatenate([deq_q[t], deq_k[t]], axis=0)
        # E4M3 half step of the element (1/16 relative, 2^-10 absolute in the
        # subnormal range) + bf16 roundings and the float32 angle (<= 2% of |z|)
        tol = np.maximum(np.abs(rot) / 16, 2.0 ** -10) + 0.02 * mag
        worst = max(worst, float((np.abs(got - rot) / tol).max()))
    assert worst <= 1.0, worst


def test_rmsnorm_unit_rms_and_zero_head():
    cfg, inp = _small(rope_theta=0.0)
    qkv = inp["qkv"].copy()
    qkv[0, QCOL + 5 * D:QCOL + 6 * D] = 0  # an all-zero q head
    inp = dict(inp, qkv=qkv)
    q8, k, _, _ = _run(cfg, inp)
    assert np.all(q8[0, 5] == 0)
    deq = oracle.e4m3_value(q8).reshape(-1, D)
    rms = np.sqrt((deq ** 2).mean(axis=1))
    live = rms > 0
    assert np.all(np.abs(rms[live] - 1.0) < 0.06)
    # scale invariance: doubling the head leaves the normalised codes unchanged
    qkv2 = inp["qkv"].copy()
    x = oracle.bf16_value(qkv2[:, : (HQ + HKV) * D]) * 2.0
    qkv2[:, : (HQ + HKV) * D] = oracle.bf16_bits(x)
    q8b, kb, _, _ = _run(cfg, dict(inp, qkv=qkv2))
    same = np.mean(q8b == q8)
    assert same > 0.999  # only eps (1e-5) separates them


def test_scaled_path_halving_scale_doubles_values():
    """k_scale = v_scale = 0.5: stored values are exactly twice the unscaled ones,
    i.e. every normal, unsaturated E4M3 code moves up one exponent step (+8)."""
    cfg, inp = _small()
    q_a, k_a, v_a, _ = _run(cfg, inp)
    cfg_s = dict(cfg, kv_scale=0.5)
    inp_s = dict(inp, k_scale=np.float32(0.5), v_scale=np.float32(0.5))
    q_b, k_b, v_b, _ = _run(cfg_s, inp_s)
    assert np.array_equal(q_a, q_b)  # q never scaled
    loc = inp["cache_loc"]
    for a, b in ((k_a, k_b), (v_a, v_b)):
        ca = a.reshape(-1, HKV * D)[loc].astype(int)
        cb = b.reshape(-1, HKV * D)[loc].astype(int)
        e = (ca >> 3) & 15
        normal = (e >= 1) & (e <= 13)
        assert normal.sum() > 100
        assert np.array_equal(cb[normal], ca[normal] + 8)


# ---- the scaled cache path, from its definition ------------------------------
# "012-attention-local-splits.py", `_prepare_qkv`, `if SCALED:`: the normalised
# (and rotated) key is divided by k_scale and cast to bf16, the raw value by
# v_scale and cast to bf16, then both are stored as E4M3. The pin computes the
# stored codes independently: float32 IEEE division (numpy), bf16 by torch's
# cast, E4M3 by brute-force nearest-code search. Non-power-of-two scales, k_scale
# != v_scale, and values chosen so that the bf16 cast before E4M3 changes the
# code (double rounding), so that a swapped divisor or a dropped bf16 cast fails.
# (A scale of 0.75 cannot show the double rounding: 4v/3 of a bf16 v never lies
# within half a bf16 step of an E4M3 rounding midpoint without being one, so
# that divisor could not tell a dropped bf16 cast apart.)

K_SCALE, V_SCALE = np.float32(0.7), np.float32(0.6)


def _e4m3_brute(vals):
    from test_oracle_formats import _brute_force_code, _e4m3_table
    codes, table = _e4m3_table()
    return np.array([_brute_force_code(float(v), codes, table) for v in np.ravel(vals)], np.uint8)


def _bf16(x):
    """float32 -> bf16 (torch's round-to-nearest-even cast) -> float64."""
    t = torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16)
    return t.to(torch.float64).numpy()


def _stored(x, scale):
    """The definition: E4M3(bf16(float32(x / scale)))."""
    q = np.asarray(x, np.float32) / np.float32(scale)  # one IEEE float32 division
    return _e4m3_brute(_bf16(q))


def _double_rounding_values(lo, hi, scale):
    """bf16 values in [lo, hi) whose E4M3 code changes when the float32 quotient
    is cast to bf16 first (and the rest, for filler)."""
    bits = np.arange(0x3C00, 0x4100, dtype=np.uint16)  # bf16 patterns of [2^-7, 8)
    v = oracle.bf16_value(bits)
    v = v[(v >= lo) & (v < hi)]
    q = (v.astype(np.float32) / np.float32(scale)).astype(np.float32)
    sens = _e4m3_brute(_bf16(q)) != _e4m3_brute(q)
    return v[sens], v[~sens]


def _unit_rms_head(payload, rng):
    """A bf16 head of 64 values: `payload` (62 values) and two values that bring
    the mean square within 1e-4 of 1, so that the normalised head equals the head
    itself (x * rsqrt(ms + 1e-5) differs from x by < 1.1e-4 relative, far inside
    half a bf16 step: the bf16 rounding returns x)."""
    assert len(payload) == 62
    r = 64.0 - float(np.sum(np.asarray(payload) ** 2))
    assert r > 1.0
    cand = oracle.bf16_value(np.arange(0x3C00, 0x4100, dtype=np.uint16))
    cand = cand[cand * cand < r]
    best = None
    for a in cand:
        b = float(_bf16(np.array([np.sqrt(r - a * a)], np.float32))[0])
        err = abs(a * a + b * b - r)
        if best is None or err < best[0]:
            best = (err, a, b)
    _, a, b = best
    head = np.concatenate([payload, [a, -b]])
    rng.shuffle(head)
    ms = float(np.mean(head ** 2))
    assert abs(ms - 1.0) <= 1e-4, ms
    return head


def test_scaled_cache_codes_from_the_definition():
    rng = np.random.default_rng(11)
    cfg = W.config("tiny_sliding_decode", batch=1, seq=("list", [37]), rope_theta=0.0, kv_scale=0.7,
                   k_scale=float(K_SCALE), v_scale=float(V_SCALE))
    inp = W.generate(cfg)
    assert inp["k_scale"] == K_SCALE and inp["v_scale"] == V_SCALE
    ks_sens, ks_rest = _double_rounding_values(0.25, 0.95, K_SCALE)
    vs_sens, vs_rest = _double_rounding_values(0.05, 6.0, V_SCALE)
    assert len(ks_sens) >= 4 and len(vs_sens) >= 8, (len(ks_sens), len(vs_sens))
    qkv = inp["qkv"].copy()
    k_heads, v_heads = [], []
    for g in range(HKV):
        pick = np.concatenate([ks_sens[g::2], rng.choice(ks_rest, 62 - len(ks_sens[g::2]), replace=False)])
        pick = pick * rng.choice([-1.0, 1.0], size=62)
        k_heads.append(_unit_rms_head(pick, rng))
        vv = np.concatenate([vs_sens[g::2][:40], rng.choice(vs_rest, 64 - len(vs_sens[g::2][:40]), replace=False)])
        v_heads.append(vv * rng.choice([-1.0, 1.0], size=64))
    for g in range(HKV):
        qkv[0, KCOL + g * D:KCOL + (g + 1) * D] = oracle.bf16_bits(k_heads[g])
        qkv[0, VCOL + g * D:VCOL + (g + 1) * D] = oracle.bf16_bits(v_heads[g])
    inp = dict(inp, qkv=qkv)
    _, k, v, skipped = _run(cfg, inp)
    assert skipped == 0
    row = int(inp["cache_loc"][0])
    got_k = k.reshape(-1, HKV * D)[row].reshape(HKV, D)
    got_v = v.reshape(-1, HKV * D)[row].reshape(HKV, D)
    for g in range(HKV):
        assert np.array_equal(got_k[g], _stored(k_heads[g], K_SCALE)), f"k head {g}"
        assert np.array_equal(got_v[g], _stored(v_heads[g], V_SCALE)), f"v head {g}"
    # the unscaled path stores E4M3(x) for the same heads (the normalised k head is x)
    _, k1, v1, _ = _run(dict(cfg, kv_scale=1.0), dict(inp, k_scale=np.float32(1), v_scale=np.float32(1)))
    for g in range(HKV):
        assert np.array_equal(k1.reshape(-1, HKV * D)[row].reshape(HKV, D)[g], _e4m3_brute(k_heads[g]))
        assert np.array_equal(v1.reshape(-1, HKV * D)[row].reshape(HKV, D)[g], _e4m3_brute(v_heads[g]))


# ---- q_norm 1: the vLLM qk_norm with the query factor folded into q ----------
# The vLLM CuTeDSL `qk_norm` page (`QKNormDirectKernel.kernel`: y = x * rstd in
# float32, y = y * scale in float32, then the store to the output dtype is the
# only rounding). The pin evaluates that chain in exact rational arithmetic:
# rstd = the float32 nearest to 1/sqrt(mean(x^2) + eps) (80-digit decimal),
# each product the float32 nearest to the exact product, then bf16 nearest
# even, then E4M3 by brute-force nearest code; no bf16 value in between.

def _rne_f32(fr):
    """The float32 nearest to the rational `fr` (ties to the even significand)."""
    from fractions import Fraction
    f = np.float32(float(fr))
    cands = [np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))]
    return min(cands, key=lambda c: (abs(Fraction(float(c)) - fr), int(np.array(c, np.float32).view(np.uint32)) & 1))


def _rstd_f32(x):
    """float32 nearest to 1/sqrt(mean(x^2) + eps32), from 80-digit decimals."""
    import decimal
    from fractions import Fraction
    ms = sum(Fraction(float(v)) ** 2 for v in x) / len(x) + Fraction(float(np.float32(1e-5)))
    with decimal.localcontext() as ctx:
        ctx.prec = 80
        r = decimal.Decimal(1) / (decimal.Decimal(ms.numerator) / decimal.Decimal(ms.denominator)).sqrt()
    return _rne_f32(Fraction(r))


def _folded_q_codes(x, s, bf16_between=False):
    from fractions import Fraction
    inv = Fraction(float(_rstd_f32(x)))
    s = Fraction(float(np.float32(s)))
    y2 = []
    for v in x:
        y1 = _rne_f32(Fraction(float(v)) * inv)
        if bf16_between:  # the mistake the pin must catch: a bf16 value before the scale
            y1 = np.float32(_bf16(np.array([y1], np.float32))[0])
        y2.append(_rne_f32(Fraction(float(y1)) * s))
    return _e4m3_brute(_bf16(np.array(y2, np.float32)))


def test_folded_q_norm_is_one_bf16_rounding_of_the_float32_chain():
    cfg = W.config("tiny_sliding_decode", rope_theta=0.0, q_norm=1)
    inp = W.generate(cfg)
    q8, k8, _, _ = _run(cfg, inp)
    sensitive = 0
    for t in range(q8.shape[0]):
        for h in range(0, HQ, 3):
            x = oracle.bf16_value(inp["qkv"][t, QCOL + h * D:QCOL + (h + 1) * D])
            want = _folded_q_codes(x, cfg["qk_scale_factor"])
            assert np.array_equal(q8[t, h], want), (t, h)
            sensitive += int(np.sum(_folded_q_codes(x, cfg["qk_scale_factor"], bf16_between=True) != want))
    assert sensitive >= 4  # the inputs tell a bf16 value before the scale apart
    # k heads are normed with scale 1: the cache rows equal q_norm 0's
    _, k0, _, _ = _run(dict(cfg, q_norm=0), inp)
    assert np.array_equal(k8, k0)
