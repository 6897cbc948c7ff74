"""Benchmark of the paged-FP8 gated attention block on GB300.

One step = the whole block over one batch of a workload. The headline line is
the largest workload that fits one GPU, the mixed full-attention decode batch:
B=256, L=1, Hq=16, Hkv=2, d=64, seq_lens log-uniform in [1, 131072], page_size
1, window 0 (no RoPE), kv_scale 1 (synthetic, seeded; about 0.73 GB of KV rows
per step). The same line carries, under "workloads", the same measurements for
the other workloads (tiny sliding decode, sliding decode, full decode at 32k,
verify block, and the extend batch of ragged prefill/extend requests, whose
roofline is the tensor peak); --workload picks another headline and
--no-others drops the rest.

The timed step is okc_attn_step in the form its plan chooses (one fused kernel
or prepare, decode and combine: the entry's config.path says which). --path
three_call times okc_prepare_qkv -> okc_attn_decode ->
okc_attn_combine_normgate instead, and the headline's "compare" entry times
the other path the same way.

Timing: W warm-up steps, then exactly K steps, replayed from CUDA graphs of
the step's launches; consecutive steps rotate over independent copies of the
inputs (cache pools, page tables, qkv) whose total exceeds 3x the L2 cache, so
every step streams its KV rows from HBM. CUDA events on the launching stream,
a device synchronize and a barrier on both sides, max over ranks. The step's
dominant kernel is then timed alone (launches without programmatic overlap)
for the roofline. `e2e` repeats the step through the public API from pinned
host buffers: per step the plan, the step's inputs moved from host memory to
the GPU (read in place by the kernels over the host link: the buffers are
page-locked and mapped), the step's calls and the output written back to host
memory.

cpu_baseline: the CPU oracle as it stands on a bounded sample of each workload
(a uniform sample of its query rows, token x head), single-threaded and on all
host cores (one thread per core, each running the oracle's attention on its own
share of the requests; ctypes calls release the interpreter lock), with the
core count and CPU model.
--impl reference times that oracle alone, on all host cores, as the reference
arm. Multi-GPU: replicas only (each rank runs its own independent batch).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import threading
import time
from concurrent.futures import ThreadPoolExecutor

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "decode tokens/s and KV-stream HBM GB/s (fraction of GB300 peak) per step"
# DRAM bytes (read + write) per launch of a step's dominant kernel, from one ncu
# capture of that kernel on that workload (dram__bytes_read.sum +
# dram__bytes_write.sum); a kernel changed since its capture has no entry.
NCU_TRAFFIC = {
    ("mixed_full_decode", "decode_kernel<fused step>"): 804015616 + 7570688,
    ("sliding_decode", "decode_kernel<fused step>"): 33093888 + 2304,
    ("full_decode_32k", "decode_kernel"): 545539072 + 2930688,
    ("verify_block", "decode_tc_kernel"): 17208832 + 0,
    ("extend", "decode_tc_kernel"): 36384768 + 247296,
}
WORKLOAD = "mixed_full_decode"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def _q_lens(cfg, seq_lens, q_lens):
    return np.full(len(seq_lens), cfg["q_len"], np.int64) if q_lens is None else np.asarray(q_lens, np.int64)


def kv_bytes(cfg, seq_lens, q_lens=None) -> int:
    """Algorithmic KV-stream bytes of one step: each request's visible keys (the
    union over its new tokens' windows) read once, K and V rows of Hkv x 64 E4M3
    bytes. q_lens: new tokens per request (default q_len each)."""
    ql = _q_lens(cfg, seq_lens, q_lens)
    w = cfg["window"]
    n = np.asarray(seq_lens, np.int64) + ql
    if w > 0:
        n = np.minimum(n, w + ql - 1)
    n = np.where(ql > 0, n, 0)
    return int(n.sum()) * cfg["num_kv_heads"] * cfg["head_dim"] * 2


def page_table_bytes_read(cfg, seq_lens, q_lens=None) -> int:
    """Bytes of page-table entries one step reads: for each request the pages
    that hold its visible keys (the union over its new tokens' windows), 4
    bytes each."""
    ql = _q_lens(cfg, seq_lens, q_lens)
    w, P = cfg["window"], cfg["page_size"]
    hi = np.asarray(seq_lens, np.int64) + ql
    n = np.minimum(hi, w + ql - 1) if w > 0 else hi
    lo = hi - n
    pages = np.where((ql > 0) & (n > 0), (hi - 1) // P - lo // P + 1, 0)
    return int(pages.sum()) * 4


def token_keys(cfg, seq_lens, q_lens=None) -> np.ndarray:
    """Per request: the sum over its new tokens of the keys each token sees."""
    ql = _q_lens(cfg, seq_lens, q_lens)
    w = cfg["window"]
    out = np.zeros(len(ql), np.int64)
    for b, (s0, q) in enumerate(zip(np.asarray(seq_lens, np.int64), ql)):
        k = s0 + np.arange(1, q + 1, dtype=np.int64)  # token i sees keys 0 .. s0 + i
        out[b] = int(np.minimum(k, w).sum()) if w > 0 else int(k.sum())
    return out


def attention_flops(cfg, seq_lens, q_lens=None) -> int:
    """Algorithmic flops of step 4: every query row (token x q head) takes a
    64-wide dot product (QK) and a 64-wide multiply-add (PV) per visible key."""
    return int(token_keys(cfg, seq_lens, q_lens).sum()) * 4 * cfg["head_dim"] * cfg["num_q_heads"]


def measured_peak_hbm():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def measured_peak_tensor():
    """Dense tensor peak of step 4's contractions, TFLOP/s: QK in E4M3 (twice the
    bf16 rate, the nominal fp8 : bf16 ratio) and PV in f16 (the bf16 rate), equal
    flops each, so time at peak is F/2 / (2P) + F/2 / P and the combined peak
    4P/3, P the measured dense bf16 rate (burst: the kernel is timed alone)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            v = float(json.load(f)["bf16_tflops"])
        return v * 4.0 / 3.0, "measured bf16 x 4/3"
    except Exception:
        return FALLBACK_BF16_TFLOPS * 4.0 / 3.0, "fallback bf16 x 4/3"


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or "unknown"."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed loop runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = [l.split(", ") for (t, l) in self.lines if t0 - 0.05 <= t <= t1 + 0.15]
        if not rows:  # a short timed region: use every sample of the run
            rows = [l.split(", ") for (_, l) in self.lines]
        sm = [float(r[1]) for r in rows if len(r) >= 9 and r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if len(r) >= 9 and r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            if len(r) >= 9:
                for n, v in zip(names, r[5:9]):
                    if v.strip().lower() == "active":
                        reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": float(max(mx)) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ---- replicas (N > 1): each rank runs its own independent batch; no data-path collective
def rank_seed(seed: int, rank: int) -> int:
    """Seed of rank `rank`'s batch: independent requests per replica."""
    return seed + 7919 * rank


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest of every rank's x (the slowest replica's time); x itself at world 1."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank: int, world: int, ms_per_step: float) -> float:
    """Whole-job tokens/s: every replica's tokens over the slowest replica's step time."""
    return tokens_per_rank * world / (ms_per_step * 1e-3)


# ------------------------------------------------------------ CPU oracle timing

def _requests(cfg, inp, bs):
    """The step restricted to requests `bs`, sharing the caches (any q lengths)."""
    bs = np.asarray(bs, np.int64)
    cu = inp["cu_seqlens_q"].astype(np.int64)
    ql = cu[bs + 1] - cu[bs]
    rows = np.concatenate([np.arange(cu[b], cu[b + 1]) for b in bs]) if len(bs) else np.zeros(0, np.int64)
    c = dict(cfg, batch=len(bs))
    d = dict(inp, qkv=inp["qkv"][rows], positions=inp["positions"][rows], cache_loc=inp["cache_loc"][rows],
             cache_seqlens=inp["cache_seqlens"][bs], seq_lens=inp["seq_lens"][bs],
             page_table=np.ascontiguousarray(inp["page_table"][bs]),
             cu_seqlens_q=np.concatenate([[0], np.cumsum(ql)]).astype(np.int32))
    return c, d, rows


class OracleRunner:
    """The oracle's step (prepare, attention, norm-gate: the functions as they
    stand) on the whole workload, its attention and norm-gate on a uniform
    sample of `frac` of the query rows (token x head; all rows at 1), spread
    over `threads` host threads (requests grouped by cost, each thread a share
    of similar cost). Caches are copied once, outside every timing: the prepare
    step rewrites the same rows with the same codes each pass."""

    def __init__(self, cfg, inp, frac=1.0, seed=0):
        import oracle
        self.o = oracle
        self.c, self.d = cfg, inp
        self.k = inp["k_cache"].copy()
        self.v = inp["v_cache"].copy()
        T, hq = inp["qkv"].shape[0], cfg["num_q_heads"]
        self.mask = None
        if frac < 1.0:
            self.mask = (np.random.default_rng(seed).random((T, hq)) < frac).astype(np.uint8)
        self.rows = T * hq if self.mask is None else int(self.mask.sum())
        self.cost = token_keys(cfg, inp["seq_lens"], inp["q_lens"]) * frac

    def groups(self, threads):
        order = np.argsort(-self.cost, kind="stable")
        load = np.zeros(threads)
        groups = [[] for _ in range(threads)]
        for b in order:
            i = int(np.argmin(load))
            groups[i].append(int(b))
            load[i] += self.cost[b]
        return [sorted(g) for g in groups if g]

    def run(self, threads=1, pool=None):
        o, c, d = self.o, self.c, self.d
        q8, _ = o.prepare(c, d, self.k, self.v)
        if threads == 1 or pool is None:
            out, _ = o.attention(c, d, q8, self.k, self.v, self.mask)
        else:
            out = np.zeros((q8.shape[0], c["num_q_heads"], 64), np.float64)

            def part(g):
                cg, dg, rows = _requests(c, d, g)
                m = None if self.mask is None else np.ascontiguousarray(self.mask[rows])
                og, _ = o.attention(cg, dg, np.ascontiguousarray(q8[rows]), self.k, self.v, m)
                out[rows] = og
            list(pool.map(part, self.groups(threads)))
        return o.normgate(c, out, d["qkv"], d.get("norm_weight"), d["eps"], self.mask)


def oracle_sample_fraction(cfg, inp, seconds: float) -> float:
    """The fraction of query rows the single-threaded oracle computes in about
    `seconds`, from a timed probe (after a warm pass) on a small uniform sample."""
    rows_all = inp["qkv"].shape[0] * cfg["num_q_heads"]
    key_rows = float(token_keys(cfg, inp["seq_lens"], inp["q_lens"]).sum()) * cfg["num_q_heads"]
    frac = min(1.0, 2.0e6 / max(key_rows, 1.0))
    probe = OracleRunner(cfg, inp, frac, seed=1)
    probe.run()  # load and warm the library
    t0 = time.perf_counter()
    probe.run()
    el = max(time.perf_counter() - t0, 1e-6)
    rows_per_s = probe.rows / el  # query rows of the workload's mix per second
    return float(min(1.0, seconds * rows_per_s / rows_all))


def cpu_oracle_baseline(cfg, inp, budget_s: float) -> dict:
    """The oracle as it stands on a bounded sample of the workload (a uniform
    sample of its query rows): tokens/s single-threaded and on all host cores."""
    B = cfg["batch"]
    cores = host_cores()
    frac = oracle_sample_fraction(cfg, inp, 0.5 * budget_s)
    r = OracleRunner(cfg, inp, frac)
    t0 = time.perf_counter()
    r.run()
    single_s = time.perf_counter() - t0
    with ThreadPoolExecutor(max_workers=cores) as pool:
        r.run(cores, pool)  # warm the threads
        reps, el = 0, 0.0
        while reps < 1 or (el < 0.25 * budget_s and reps < 1000):
            t0 = time.perf_counter()
            r.run(cores, pool)
            el += time.perf_counter() - t0
            reps += 1
    toks = r.rows / cfg["num_q_heads"]  # query rows counted as tokens
    what = "all" if frac >= 1.0 else f"{100.0 * frac:.3g}% (uniform sample)"
    return {"value": toks / single_s, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{what} of the query rows of {B} requests of {cfg['name']} (one pass), single-threaded C oracle",
            "seconds": single_s,
            "all_cores": {"value": toks * reps / el, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                          "sample": f"the same rows x {reps} pass(es), attention spread over {cores} host threads",
                          "seconds": el},
            "nproc": cores, "cpu_model": cpu_model()}


def run_reference(args, world, rank):
    """The reference arm: the CPU oracle as it stands, on all host cores, each of
    the K steps one bounded sample (a uniform sample of the query rows) of the
    same workload."""
    if rank != 0:
        return
    cfg = W.config(args.workload)
    inp = W.generate(cfg)
    B, L = cfg["batch"], cfg["q_len"]
    cores = host_cores()
    total_budget = 60.0  # seconds of oracle work (all cores) for the whole run
    frac = oracle_sample_fraction(cfg, inp, total_budget * cores / max(1, args.steps + args.warmup))
    r = OracleRunner(cfg, inp, frac)
    el = 0.0
    with ThreadPoolExecutor(max_workers=cores) as pool:
        for _ in range(args.warmup):
            r.run(cores, pool)
        for _ in range(args.steps):
            t0 = time.perf_counter()
            r.run(cores, pool)
            el += time.perf_counter() - t0
    toks = r.rows / cfg["num_q_heads"]
    value = toks * args.steps / el
    T = inp["qkv"].shape[0]
    what = "all" if frac >= 1.0 else f"{100.0 * frac:.3g}% (uniform sample)"
    sample = (f"{what} of the query rows of {args.workload} per step, C oracle with its attention spread over "
              f"{cores} host threads ({cpu_model()})")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * T / value,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": {"workload": args.workload, "batch": B, "q_len": L, "page_size": cfg["page_size"],
                   "window": cfg["window"], "rope_theta": cfg["rope_theta"]},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------- GPU measurement

class Bench:
    """Shared state of one bench run on one GPU."""

    def __init__(self, args, world, rank, local):
        import torch
        import fp8_kv_paged_gb300 as okc
        self.torch, self.okc = torch, okc
        self.args, self.world, self.rank = args, world, rank
        self.dev = torch.device("cuda", local)
        self.stream = torch.cuda.Stream(device=self.dev)
        self.l2 = torch.cuda.get_device_properties(self.dev).L2_cache_size

    def barrier(self):
        self.torch.cuda.synchronize(self.dev)
        if self.world > 1:
            self.torch.distributed.barrier()

    def capture(self, fn, nsteps):
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(self.stream):
            fn(0)  # warm the launch path
        self.stream.synchronize()
        with torch.cuda.graph(g, stream=self.stream):
            for i in range(nsteps):
                fn(i)
        return g

    def timed(self, fn, steps_total, warm, R):
        """ms per step of `steps_total` steps replayed from graphs (exact count)."""
        torch = self.torch
        r_, m_ = divmod(steps_total, R)
        g_main = self.capture(fn, R) if r_ else None
        g_rem = self.capture(fn, m_) if m_ else None
        nw = max(3, min(warm, R))
        g_warm = self.capture(fn, nw)
        left = warm
        while left > 0:
            g_warm.replay()
            left -= nw
        self.barrier()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        w0 = time.time()
        with torch.cuda.stream(self.stream):
            ev0.record(self.stream)
            for _ in range(r_):
                g_main.replay()
            if g_rem is not None:
                g_rem.replay()
            ev1.record(self.stream)
        self.barrier()
        w1 = time.time()
        ms = max_over_ranks(ev0.elapsed_time(ev1), self.world, self.dev)
        return ms / steps_total, w0, w1

    def measure(self, name, steps, warmup, clocks=None, compare=False, cpu=True):
        """Every figure of one workload: the step, its dominant kernel alone, e2e, CPU baseline."""
        torch, okc, args, dev, stream = self.torch, self.okc, self.args, self.dev, self.stream
        cfg = W.config(name)
        inp = W.generate(cfg, seed=rank_seed(cfg["seed"], self.rank))
        T = inp["qkv"].shape[0]
        ql = inp["q_lens"] if "q_lens" in cfg else None  # per-request q lengths (prefill/extend)
        kvb = kv_bytes(cfg, inp["seq_lens"], ql)
        flops = attention_flops(cfg, inp["seq_lens"], ql)

        # independent input sets so that consecutive steps miss in L2
        base = W.to_torch(inp, dev)
        if cfg["rope_theta"] != 0.0:
            npos = int(inp["positions"].max()) + 1
            base["rope_table"] = torch.empty((npos, 64), dtype=torch.float32, device=dev)
            okc.okc_rope_table_init(cfg["rope_theta"], npos, base["rope_table"])
        set_bytes = sum(t.numel() * t.element_size() for k, t in base.items()
                        if t is not None and k not in ("rope_table",))
        n_sets = max(2, math.ceil(3 * self.l2 / set_bytes))
        shared = ("rope_table", "k_scale", "v_scale", "norm_weight")
        sets = [base] + [{k: (None if t is None else (t if k in shared else t.clone())) for k, t in base.items()}
                         for _ in range(n_sets - 1)]
        plan_opts = {}
        if args.chunk_keys:
            plan_opts["chunk_keys"] = args.chunk_keys
        if args.step_form != "plan":
            plan_opts["flags"] = okc.PLAN_STEP_ONE_LAUNCH if args.step_form == "one" else \
                okc.PLAN_STEP_THREE_LAUNCHES
        if args.early_gather:
            plan_opts["flags"] = plan_opts.get("flags", 0) | okc.PLAN_EARLY_GATHER
        plan_opts = plan_opts or None
        step = okc.AttnStep(cfg, inp["seq_lens"], opts=plan_opts, q_lens=ql)
        fused = args.path == "fused"

        def run_step(st, s_, use_fused):
            if use_fused:
                st.run_fused(s_, eps=inp["eps"], stream=stream)
            else:
                st.run(s_, eps=inp["eps"], stream=stream)

        R = n_sets * max(1, 48 // n_sets)  # steps per graph replay
        if clocks is not None:
            clocks.start()
            time.sleep(0.3)
        ms_step, t_wall0, t_wall1 = self.timed(lambda i: run_step(step, sets[i % n_sets], fused), steps, warmup, R)

        # the step's dominant kernel alone, no programmatic overlap: the fused
        # step kernel, or the decode kernel of the three-call path
        step_np = okc.AttnStep(cfg, inp["seq_lens"],
                               opts=dict(plan_opts or {}, flags=(plan_opts or {}).get("flags", 0) | okc.PLAN_NO_PDL),
                               q_lens=ql)
        for s_ in sets:
            step_np.run(s_, eps=inp["eps"], stream=stream)
        stream.synchronize()
        step_kernels = step.sizes["step_kernels"]
        if fused and step_kernels == 1:
            def one_kernel(i):
                s_ = sets[i % n_sets]
                okc.okc_attn_step(step_np.plan, s_["qkv"], s_["positions"], s_["cache_loc"], s_["k_cache"],
                                  s_["v_cache"], s_["k_scale"], s_["v_scale"], s_["rope_table"], s_["page_table"],
                                  s_["cache_seqlens"], s_["cu_seqlens_q"], s_["seq_lens"], s_["norm_weight"],
                                  inp["eps"], step_np.o_partial, step_np.lse_partial, step_np.out, stream)
            kname = "decode_kernel<fused step>"
        else:
            def one_kernel(i):
                s_ = sets[i % n_sets]
                okc.okc_attn_decode(step_np.plan, step_np.q_fp8, s_["k_cache"], s_["v_cache"], s_["k_scale"],
                                    s_["v_scale"], s_["page_table"], s_["cache_seqlens"], s_["cu_seqlens_q"],
                                    s_["seq_lens"], step_np.o_partial, step_np.lse_partial, stream)
            kname = "decode_tc_kernel" if cfg["q_len"] >= 2 else "decode_kernel"
        kernel_ms, _, _ = self.timed(one_kernel, max(R, min(steps, 20 * R)), 3, R)
        kernel_us = 1000.0 * kernel_ms
        clk = clocks.stop(t_wall0, t_wall1) if clocks is not None else None

        other = {}
        if compare:
            def run_other(i):
                run_step(step, sets[i % n_sets], not fused)
            oms, _, _ = self.timed(run_other, max(R, min(steps, 20 * R)), 3, R)
            other = {"path": "three_call" if fused else "fused", "ms_per_step": oms,
                     "value": job_throughput(T, self.world, oms)}

        e2e = run_e2e(cfg, inp, okc, torch, dev, stream, steps=min(max(steps, 20), 200), fused=fused)
        peak, peak_kind = measured_peak_hbm()
        tpeak, tpeak_kind = measured_peak_tensor()
        achieved = kvb / (kernel_us * 1e-6) / 1e9
        tflops = flops / (kernel_us * 1e-6) / 1e12
        # the bound: HBM while the step's flops per algorithmic KV byte stay below
        # the ratio of the two peaks (decode: 16 flop/B, verify: 128), else the
        # tensor cores (prefill/extend: thousands of flops per KV byte)
        if flops / max(kvb, 1) < tpeak * 1e12 / (peak * 1e9):
            roof = {"kernel": kname, "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                    "frac": achieved / peak, "traffic": NCU_TRAFFIC.get((name, kname)), "algorithmic_bytes": kvb,
                    "peak_source": peak_kind, "avg_launch_us": kernel_us, "tflops": tflops}
        else:
            roof = {"kernel": kname, "bound": "tensor", "achieved": tflops, "peak": tpeak, "unit": "TFLOP/s",
                    "frac": tflops / tpeak, "traffic": NCU_TRAFFIC.get((name, kname)), "algorithmic_flops": flops,
                    "algorithmic_bytes": kvb, "kv_gbs": achieved, "peak_source": tpeak_kind,
                    "avg_launch_us": kernel_us}
        res = {
            "value": job_throughput(T, self.world, ms_step), "unit": "tokens/s", "ms_per_step": ms_step,
            "config": {"workload": name, "batch": cfg["batch"], "q_len": cfg["q_len"], "tokens": T,
                       "page_size": cfg["page_size"], "window": cfg["window"], "rope_theta": cfg["rope_theta"],
                       "kv_scale": cfg["kv_scale"], "kv_bytes_per_step": kvb,
                       "path": "okc_attn_step (%d kernel%s)" % (step_kernels, "" if step_kernels == 1 else "s")
                       if fused else "three calls",
                       "num_work": step.sizes["num_work"],
                       "parallelism": "replicas" if self.world > 1 else "single-gpu",
                       "l2": "inputs rotate over %d sets (%.0f MB total > 3x L2)" % (n_sets, n_sets * set_bytes / 1e6)},
            "kv_stream_gbs_step": kvb / (ms_step * 1e-3) / 1e9,
            "kv_stream_frac_step": kvb / (ms_step * 1e-3) / 1e9 / peak,
            "roofline": roof,
            "e2e": e2e,
            "gpu_launches": (step_kernels if fused else 3) * steps,
        }
        if clk is not None:
            res["clocks"] = clk
        if other:
            res["compare"] = other
        if cpu and self.rank == 0 and not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_oracle_baseline(cfg, inp, budget_s=args.cpu_budget)
        del sets, base, step, step_np
        torch.cuda.synchronize(dev)
        torch.cuda.empty_cache()
        return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="okc", choices=["okc", "reference"])
    ap.add_argument("--workload", default=WORKLOAD, choices=list(W.WORKLOADS))
    ap.add_argument("--no-others", action="store_true", help="measure the headline workload only")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work per workload")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--path", default="fused", choices=["fused", "three_call"],
                    help="okc_attn_step or okc_prepare_qkv + okc_attn_decode + okc_attn_combine_normgate")
    ap.add_argument("--no-compare", action="store_true", help="skip timing the other path")
    ap.add_argument("--chunk-keys", type=int, default=0,
                    help="keys per split work item (plan option; 0 = the plan's heuristic)")
    ap.add_argument("--step-form", default="plan", choices=["plan", "one", "three"],
                    help="okc_attn_step as one kernel or three (plan option; default: the plan's choice)")
    ap.add_argument("--early-gather", action="store_true",
                    help="plan flag OKC_PLAN_EARLY_GATHER (consecutive steps run on different input sets)")
    args = ap.parse_args()
    world, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, world, rank)

    import torch
    import fp8_kv_paged_gb300 as okc

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    okc.build()
    b = Bench(args, world, rank, local)

    clocks = ClockSampler(local)
    head = b.measure(args.workload, args.steps, args.warmup, clocks=clocks, compare=not args.no_compare)
    others = {}
    if not args.no_others:
        for name in W.WORKLOADS:
            if name != args.workload:
                others[name] = b.measure(name, args.steps, args.warmup)
    line = {
        "metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3/f16->f32",
        "data": "synthetic (seeded); L2 defeated by rotating independent input sets > 3x L2",
    }
    line.update({k: v for k, v in head.items() if k not in ("value", "unit", "ms_per_step")})
    line["gpu_launches"] = head["gpu_launches"] + sum(o["gpu_launches"] for o in others.values())
    if others:
        line["workloads"] = others
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_e2e(cfg, inp, okc, torch, dev, stream, steps: int, fused: bool = True):
    """Per step: the plan re-made in place from the host seq_lens, the step's inputs from pinned host
    memory (okc_attn_step_host: read in place by the kernels; the three calls:
    copied to device buffers first), the step, the output back in host memory;
    K steps timed on the host clock. h2d counts the host input bytes the step
    consumes (the kernels read only the page-table entries they need)."""
    names = ("qkv", "positions", "cache_loc", "cache_seqlens", "cu_seqlens_q", "seq_lens", "page_table")
    host = W.to_torch({**inp, "k_cache": inp["k_cache"][:1], "v_cache": inp["v_cache"][:1]}, "cpu")
    pinned = {k: host[k].pin_memory() for k in names}
    dev_in = W.to_torch(inp, dev)
    if cfg["rope_theta"] != 0.0:
        npos = int(inp["positions"].max()) + 1
        dev_in["rope_table"] = torch.empty((npos, 64), dtype=torch.float32, device=dev)
        okc.okc_rope_table_init(cfg["rope_theta"], npos, dev_in["rope_table"], stream)
    T = inp["qkv"].shape[0]
    ql = inp["q_lens"] if "q_lens" in cfg else None
    out_host = torch.empty((T, cfg["num_q_heads"] * cfg["head_dim"]), dtype=torch.bfloat16).pin_memory()
    sizes = okc.okc_attn_plan_sizes(cfg, inp["seq_lens"], q_lens=ql)
    ws = torch.empty(sizes["workspace_bytes"], dtype=torch.uint8, device=dev)
    q8 = torch.empty(sizes["q_fp8_bytes"], dtype=torch.uint8, device=dev)
    op = torch.empty(max(16, sizes["o_partial_bytes"]) // 4, dtype=torch.float32, device=dev)
    lp = torch.empty(max(16, sizes["lse_partial_bytes"]) // 4, dtype=torch.float32, device=dev)
    out = torch.empty_like(out_host, device=dev)
    # the step's inputs (the page table: the entries the kernels read, the pages
    # spanning each request's visible keys; every other input whole), and the
    # plan's upload (the workspace up to its q scratch)
    h2d = sum(pinned[k].numel() * pinned[k].element_size() for k in names if k != "page_table") + \
        page_table_bytes_read(cfg, inp["seq_lens"], ql) + sizes["workspace_bytes"] - sizes["q_fp8_bytes"]
    d2h = out_host.numel() * 2

    io = okc.HostStepIO(dict(pinned, out=out_host), dict({k: dev_in[k] for k in names}, out=out))

    plan = okc.okc_attn_plan(cfg, inp["seq_lens"], ws, stream=stream, q_lens=ql)

    def one():
        plan.update(inp["seq_lens"], stream, q_lens=ql)  # the step's plan, re-made in place from the host lengths
        if fused:  # one C call: the step from host buffers, output in host memory, synchronize
            okc.okc_attn_step_host(plan, io, None, dev_in["k_cache"], dev_in["v_cache"], dev_in["k_scale"],
                                   dev_in["v_scale"], dev_in["rope_table"], dev_in["norm_weight"], inp["eps"],
                                   op, lp, stream)
            return
        for k in names:
            dev_in[k].copy_(pinned[k], non_blocking=True)
        okc.okc_prepare_qkv(plan, dev_in["qkv"], dev_in["positions"], dev_in["cache_loc"], dev_in["k_cache"],
                            dev_in["v_cache"], dev_in["k_scale"], dev_in["v_scale"], dev_in["rope_table"],
                            q8, stream)
        okc.okc_attn_decode(plan, q8, dev_in["k_cache"], dev_in["v_cache"], dev_in["k_scale"],
                            dev_in["v_scale"], dev_in["page_table"], dev_in["cache_seqlens"],
                            dev_in["cu_seqlens_q"], dev_in["seq_lens"], op, lp, stream)
        okc.okc_attn_combine_normgate(plan, op, lp, dev_in["qkv"], dev_in["norm_weight"], inp["eps"], out,
                                      stream)
        out_host.copy_(out, non_blocking=True)
        stream.synchronize()

    with torch.cuda.stream(stream):
        for _ in range(5):
            one()
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for _ in range(steps):
            one()
        el = time.perf_counter() - t0
    plan.close()
    return {"value": T * steps / el, "unit": "tokens/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": 1000.0 * el / steps, "steps": steps,
            "api": "okc_attn_plan_update + okc_attn_step_host" if fused else "okc_attn_plan_update + three calls"}


if __name__ == "__main__":
    main()
