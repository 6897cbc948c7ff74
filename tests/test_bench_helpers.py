"""bench.py's accounting without a GPU: the algorithmic KV bytes of a step equal
256 bytes per key the planner's work list covers (two independent accounts of
the visible keys), the full-context workload's bytes are exact, the page-table
bytes an end-to-end step reads are the pages the work list touches, and the clock
sampler reads nvidia-smi's CSV rows into a median SM clock, the maximum clock
and the active throttle reasons of the timed region."""
import time

import numpy as np

import bench
import fp8_kv_paged_gb300 as okc
import workloads as W

HOST = {"sm_count": 152, "ctas_per_sm": 3}


def test_kv_bytes_equal_the_keys_the_work_list_covers():
    okc.build()
    for name in W.DECODE_WORKLOADS:
        cfg = W.config(name)
        seq = W.lengths(cfg)
        items = okc.okc_attn_plan_items(cfg, seq, HOST)
        covered = int((items[:, 2].astype(np.int64) - items[:, 1]).sum())
        assert bench.kv_bytes(cfg, seq) == covered * 2 * 64 * 2, name
    cfg = W.config("full_decode_32k")
    assert bench.kv_bytes(cfg, W.lengths(cfg)) == 64 * 32769 * 256


def test_page_table_bytes_are_the_pages_the_work_list_touches():
    """The end-to-end host-to-device count takes the page-table entries the step
    reads: 4 bytes per distinct page holding a key of some work item."""
    okc.build()
    for name in W.DECODE_WORKLOADS:
        cfg = W.config(name)
        seq = W.lengths(cfg)
        items = okc.okc_attn_plan_items(cfg, seq, HOST)
        P = cfg["page_size"]
        it = items[np.lexsort((items[:, 1], items[:, 0]))].astype(np.int64)
        first, last = it[:, 1] // P, (it[:, 2] - 1) // P
        count = int((last - first + 1).sum())
        # a page shared by consecutive items of one request is counted once
        same = (it[1:, 0] == it[:-1, 0]) & (first[1:] <= last[:-1])
        count -= int((last[:-1][same] - first[1:][same] + 1).sum())
        assert bench.page_table_bytes_read(cfg, seq) == 4 * count, name


def test_extend_accounting():
    """The extend workload: the algorithmic KV bytes are each request's visible
    keys once (seq + q_len on a full-attention layer); the flops count every
    token's visible keys; the work list covers each query block's keys once
    (blocks of 16 tokens on the tcgen05 kernel)."""
    okc.build()
    cfg = W.config("extend")
    inp = W.generate(cfg)
    seq, ql = inp["seq_lens"].astype(np.int64), inp["q_lens"].astype(np.int64)
    assert bench.kv_bytes(cfg, inp["seq_lens"], inp["q_lens"]) == int((seq + ql).sum()) * 256
    keys = sum(int((s + np.arange(1, q + 1)).sum()) for s, q in zip(seq, ql))
    assert bench.attention_flops(cfg, inp["seq_lens"], inp["q_lens"]) == keys * 4 * 64 * 16
    items = okc.okc_attn_plan_items_varlen(cfg, inp["seq_lens"], inp["q_lens"], {"sm_count": 152, "ctas_per_sm": 1})
    covered = int((items[:, 3].astype(np.int64) - items[:, 2]).sum())
    want = sum(int(s + min(i + 16, q)) for s, q in zip(seq, ql) for i in range(0, q, 16))
    assert covered == want


class _FakeProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def test_clock_sampler_parses_rows_of_the_timed_region():
    s = bench.ClockSampler(0)
    s.proc = _FakeProc()
    t0 = time.time()
    row = "0, {sm}, 2070, 900.5, 0x0, {hw}, Not Active, Not Active, {cap}"
    s.lines = [(t0 - 5.0, row.format(sm=1000, hw="Active", cap="Not Active")),  # before the region
               (t0 + 0.01, row.format(sm=2070, hw="Not Active", cap="Not Active")),
               (t0 + 0.02, row.format(sm=2055, hw="Not Active", cap="Active")),
               (t0 + 0.03, row.format(sm=2070, hw="Not Active", cap="Not Active"))]
    r = s.stop(t0, t0 + 0.05)
    assert r["samples"] == 3 and r["sm_mhz"] == 2070.0 and r["sm_max_mhz"] == 2070.0
    assert r["reasons"] == ["sw_power_cap"]  # the hw_slowdown row lies outside the region
    s2 = bench.ClockSampler(0)
    assert s2.stop(t0, t0 + 1)["reasons"] == ["nvidia-smi unavailable"]
