"""The C-ABI library builds for sm_103a, loads, exports every entry point the
header declares, and rejects bad arguments on the host before any GPU work."""
import ctypes
import os
import re

import pytest

import fp8_kv_paged_gb300 as okc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "okc_attn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(okc_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    okc.build()
    return okc.load()


def test_header_declares_the_four_steps():
    names = _declared()
    for n in ("okc_attn_plan", "okc_prepare_qkv", "okc_attn_decode", "okc_attn_combine_normgate"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert names
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(okc.EXPORTED_SYMBOLS) == names


def test_status_strings(lib):
    for s in range(5):
        assert okc.load().okc_status_string(s)


def _cfg(**kw):
    c = dict(batch=2, q_len=1, num_q_heads=16, num_kv_heads=2, head_dim=64, page_size=1,
             window=2048, max_pages=512, num_pages=1024, rope_theta=5e5, qk_scale_factor=5.473,
             sm_scale=0.125, kv_scale=1.0)
    c.update(kw)
    return c


@pytest.mark.parametrize("bad,status", [
    (dict(head_dim=128), okc.ERR_UNSUPPORTED),
    (dict(num_q_heads=32), okc.ERR_UNSUPPORTED),
    (dict(page_size=3), okc.ERR_UNSUPPORTED),
    (dict(q_len=0), okc.ERR_INVALID),
    (dict(q_len=65537), okc.ERR_INVALID),
    (dict(q_norm=2), okc.ERR_INVALID),
    (dict(window=-1), okc.ERR_INVALID),
    (dict(sm_scale=0.0), okc.ERR_INVALID),
    (dict(kv_scale=-1.0), okc.ERR_INVALID),
    (dict(rope_theta=float("nan")), okc.ERR_INVALID),
    (dict(num_q_heads=15), okc.ERR_INVALID),
    (dict(batch=(1 << 22) + 1, q_len=16), okc.ERR_UNSUPPORTED),  # 2^26 tokens + 16
    (dict(max_pages=(1 << 30) + 1), okc.ERR_UNSUPPORTED),
])
def test_bad_config_rejected_before_gpu_work(lib, bad, status):
    """Config validation runs first, so these need no GPU."""
    with pytest.raises(okc.OkcError) as e:
        okc.okc_attn_plan_sizes(_cfg(**bad), [100, 300])
    assert e.value.status == status


def test_null_arguments_rejected(lib):
    P = ctypes.c_void_p
    assert lib.okc_attn_plan_sizes(None, None, None, None) == okc.ERR_INVALID
    assert lib.okc_attn_plan_destroy(None) == okc.OK
    assert lib.okc_prepare_qkv(None, *([None] * 8), 0, None, None) == okc.ERR_INVALID
    assert lib.okc_attn_decode(None, *([None] * 12)) == okc.ERR_INVALID
    assert lib.okc_attn_combine_normgate(None, None, None, None, None, 1e-5, None, None) == okc.ERR_INVALID
    assert lib.okc_rope_table_init(5e5, 0, None, None) == okc.ERR_INVALID
    v = ctypes.c_uint32()
    assert lib.okc_attn_plan_read_errors(None, None, ctypes.byref(v)) == okc.ERR_INVALID
    # the bounded-wait diagnostic checks its arguments before any GPU work
    assert lib.okc_selftest_bounded_wait(None, 1000, None) == okc.ERR_INVALID
    dummy = ctypes.c_uint32()
    assert lib.okc_selftest_bounded_wait(ctypes.byref(dummy), 0, None) == okc.ERR_INVALID
    assert lib.okc_selftest_bounded_wait(ctypes.byref(dummy), 1000001, None) == okc.ERR_INVALID
