"""Python binding of libokc_attn.so, the GB300 paged-FP8 gated attention block.

Argument marshalling only: every step of the block runs in the library's CUDA
kernels. Functions carry the C entry points' names (see include/okc_attn.h);
tensors are passed by device pointer, streams by handle (default: torch's
current stream). There is no CPU fallback: if the library cannot be loaded,
every call raises.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build_mod

__all__ = ["build", "load", "OkcError", "Plan", "okc_attn_plan", "okc_attn_plan_create", "okc_attn_plan_sizes",
           "okc_attn_plan_items", "okc_attn_plan_items_varlen", "okc_attn_plan_max_sizes",
           "okc_attn_plan_workspace_size",
           "okc_rope_table_init", "okc_prepare_qkv", "okc_attn_decode",
           "okc_attn_combine_normgate", "okc_attn_plan_read_errors", "okc_attn_plan_clear_errors", "AttnStep",
           "okc_attn_decode_combine_noalloc", "okc_selftest_bounded_wait", "okc_attn_step", "okc_attn_step_host", "HostStepIO", "STEP_IO",
           "DEVERR_CACHE_LOC", "DEVERR_POSITION", "DEVERR_PAGE", "DEVERR_LENGTHS", "DEVERR_TIMEOUT",
           "PLAN_NO_PDL", "PLAN_NO_TCGEN05", "PLAN_STEP_ONE_LAUNCH", "PLAN_STEP_THREE_LAUNCHES",
           "PLAN_EARLY_GATHER",
           "QNORM_BF16", "QNORM_FOLDED_SCALE",
           "EXPORTED_SYMBOLS"]

OK, ERR_INVALID, ERR_UNSUPPORTED, ERR_CUDA, ERR_WORKSPACE = 0, 1, 2, 3, 4
DEVERR_CACHE_LOC, DEVERR_POSITION, DEVERR_PAGE, DEVERR_LENGTHS, DEVERR_TIMEOUT = 0x1, 0x2, 0x4, 0x8, 0x10
PLAN_NO_PDL = 0x1
PLAN_NO_TCGEN05 = 0x2
PLAN_STEP_ONE_LAUNCH = 0x4
PLAN_STEP_THREE_LAUNCHES = 0x8
PLAN_EARLY_GATHER = 0x10
QNORM_BF16, QNORM_FOLDED_SCALE = 0, 1

EXPORTED_SYMBOLS = [
    "okc_attn_plan_sizes", "okc_attn_plan", "okc_attn_plan_destroy", "okc_attn_plan_get_sizes",
    "okc_attn_plan_read_errors", "okc_rope_table_init", "okc_prepare_qkv", "okc_attn_decode",
    "okc_attn_combine_normgate", "okc_status_string", "okc_attn_decode_combine_noalloc",
    "okc_attn_step", "okc_attn_step_host", "okc_attn_plan_items", "okc_attn_plan_update",
    "okc_attn_plan_max_sizes", "okc_attn_plan_workspace_size", "okc_attn_plan_create",
    "okc_attn_plan_scratch_sizes", "okc_selftest_bounded_wait", "okc_attn_plan_clear_errors",
    "okc_attn_plan_varlen", "okc_attn_plan_sizes_varlen", "okc_attn_plan_items_varlen",
    "okc_attn_plan_update_varlen",
]


class OkcError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _lib.okc_status_string(status).decode() if _lib is not None else str(status)
        super().__init__(f"{where}: {msg} (status {status})")


class _Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("batch", "q_len", "num_q_heads", "num_kv_heads", "head_dim", "page_size", "window",
                 "max_pages", "num_pages")] + \
               [(n, ctypes.c_float) for n in ("rope_theta", "qk_scale_factor", "sm_scale", "kv_scale")] + \
               [("q_norm", ctypes.c_int32)]


class _Options(ctypes.Structure):
    _fields_ = [("chunk_keys", ctypes.c_int32), ("flags", ctypes.c_int32),
                ("ctas_per_sm", ctypes.c_int32), ("sm_count", ctypes.c_int32), ("max_context", ctypes.c_int32)]


class _HostStep(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("qkv_host", "positions_host", "cache_loc_host", "cache_seqlens_host", "cu_seqlens_q_host",
                 "seq_lens_host", "page_table_host", "out_host", "qkv", "positions", "cache_loc",
                 "cache_seqlens", "cu_seqlens_q", "seq_lens", "page_table", "out")]


class _Sizes(ctypes.Structure):
    _fields_ = [("workspace_bytes", ctypes.c_size_t), ("q_fp8_bytes", ctypes.c_size_t),
                ("o_partial_bytes", ctypes.c_size_t), ("lse_partial_bytes", ctypes.c_size_t),
                ("num_work", ctypes.c_int32), ("num_tokens", ctypes.c_int32),
                ("max_chunks", ctypes.c_int32), ("step_kernels", ctypes.c_int32)]


_lib = None


def build(force: bool = False) -> str:
    """Compile the CUDA library for sm_103a (in-tree) and load it."""
    path = _build_mod.build(force=force)
    load(path)
    return path


def load(path: str | None = None):
    """Load libokc_attn.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or _build_mod.LIB
    if not os.path.exists(path):
        raise RuntimeError(f"libokc_attn.so is not built ({path}); call fp8_kv_paged_gb300.build()")
    lib = ctypes.CDLL(path)
    P, i32, f32, st = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_int
    lib.okc_status_string.restype = ctypes.c_char_p
    lib.okc_status_string.argtypes = [st]
    lib.okc_attn_plan_sizes.restype = st
    lib.okc_attn_plan_sizes.argtypes = [ctypes.POINTER(_Config), P, ctypes.POINTER(_Options),
                                        ctypes.POINTER(_Sizes)]
    lib.okc_attn_plan_sizes_varlen.restype = st
    lib.okc_attn_plan_sizes_varlen.argtypes = [ctypes.POINTER(_Config), P, P, ctypes.POINTER(_Options),
                                               ctypes.POINTER(_Sizes)]
    lib.okc_attn_plan_items_varlen.restype = st
    lib.okc_attn_plan_items_varlen.argtypes = [ctypes.POINTER(_Config), P, P, ctypes.POINTER(_Options), P, i32,
                                               ctypes.POINTER(ctypes.c_int32)]
    lib.okc_attn_plan_varlen.restype = st
    lib.okc_attn_plan_varlen.argtypes = [ctypes.POINTER(_Config), P, P, ctypes.POINTER(_Options), P,
                                         ctypes.c_size_t, P, ctypes.POINTER(ctypes.c_void_p)]
    lib.okc_attn_plan_update_varlen.restype = st
    lib.okc_attn_plan_update_varlen.argtypes = [P, P, P, P]
    lib.okc_attn_plan_items.restype = st
    lib.okc_attn_plan_items.argtypes = [ctypes.POINTER(_Config), P, ctypes.POINTER(_Options), P, i32,
                                        ctypes.POINTER(ctypes.c_int32)]
    lib.okc_attn_plan.restype = st
    lib.okc_attn_plan.argtypes = [ctypes.POINTER(_Config), P, ctypes.POINTER(_Options), P,
                                  ctypes.c_size_t, P, ctypes.POINTER(ctypes.c_void_p)]
    lib.okc_attn_plan_max_sizes.restype = st
    lib.okc_attn_plan_max_sizes.argtypes = [ctypes.POINTER(_Config), i32, ctypes.POINTER(_Options),
                                            ctypes.POINTER(_Sizes)]
    lib.okc_attn_plan_workspace_size.restype = st
    lib.okc_attn_plan_workspace_size.argtypes = [ctypes.POINTER(_Config), i32, ctypes.POINTER(ctypes.c_size_t)]
    lib.okc_attn_plan_create.restype = st
    lib.okc_attn_plan_create.argtypes = [ctypes.POINTER(_Config), P, P, ctypes.c_size_t, P,
                                         ctypes.POINTER(ctypes.c_void_p)]
    lib.okc_attn_plan_scratch_sizes.restype = st
    lib.okc_attn_plan_scratch_sizes.argtypes = [P, ctypes.POINTER(_Sizes)]
    lib.okc_selftest_bounded_wait.restype = st
    lib.okc_selftest_bounded_wait.argtypes = [P, i32, P]
    lib.okc_attn_plan_update.restype = st
    lib.okc_attn_plan_update.argtypes = [P, P, P]
    lib.okc_attn_plan_destroy.restype = st
    lib.okc_attn_plan_destroy.argtypes = [P]
    lib.okc_attn_plan_get_sizes.restype = st
    lib.okc_attn_plan_get_sizes.argtypes = [P, ctypes.POINTER(_Sizes)]
    lib.okc_attn_plan_clear_errors.restype = st
    lib.okc_attn_plan_clear_errors.argtypes = [P, P]
    lib.okc_attn_plan_read_errors.restype = st
    lib.okc_attn_plan_read_errors.argtypes = [P, P, ctypes.POINTER(ctypes.c_uint32)]
    lib.okc_rope_table_init.restype = st
    lib.okc_rope_table_init.argtypes = [f32, i32, P, P]
    lib.okc_prepare_qkv.restype = st
    lib.okc_prepare_qkv.argtypes = [P, P, P, P, P, P, P, P, P, i32, P, P]
    lib.okc_attn_decode.restype = st
    lib.okc_attn_decode.argtypes = [P, P, P, P, P, P, P, P, P, P, P, P, P]
    lib.okc_attn_combine_normgate.restype = st
    lib.okc_attn_combine_normgate.argtypes = [P, P, P, P, P, f32, P, P]
    lib.okc_attn_step.restype = st
    lib.okc_attn_step.argtypes = [P] * 9 + [i32] + [P] * 5 + [f32, P, P, P, P]
    lib.okc_attn_step_host.restype = st
    lib.okc_attn_step_host.argtypes = [P, ctypes.POINTER(_HostStep)] + [P] * 5 + [i32, P, f32, P, P, P]
    lib.okc_attn_decode_combine_noalloc.restype = st
    lib.okc_attn_decode_combine_noalloc.argtypes = [ctypes.POINTER(_Config), P] + [P] * 11 + [f32, P, P]
    _lib = lib
    return lib


def _check(status: int, where: str):
    if status != OK:
        raise OkcError(status, where)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return stream if isinstance(stream, int) else stream.cuda_stream


def _config(cfg: dict) -> _Config:
    return _Config(cfg["batch"], cfg["q_len"], cfg["num_q_heads"], cfg["num_kv_heads"],
                   cfg["head_dim"], cfg["page_size"], cfg["window"], cfg["max_pages"],
                   cfg["num_pages"], cfg["rope_theta"], cfg["qk_scale_factor"], cfg["sm_scale"],
                   cfg["kv_scale"], int(cfg.get("q_norm", 0)))


def _options(opts: dict | None):
    if not opts:
        return None
    return ctypes.byref(_Options(opts.get("chunk_keys", 0), opts.get("flags", 0),
                                 opts.get("ctas_per_sm", 0), opts.get("sm_count", 0),
                                 opts.get("max_context", 0)))


def _sizes_dict(z: _Sizes) -> dict:
    return {f: getattr(z, f) for f, _ in _Sizes._fields_}


def _i32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.int32)


def _data(a):
    return None if a is None else a.ctypes.data


def okc_attn_plan_sizes(cfg: dict, seq_lens_host, opts: dict | None = None, q_lens=None) -> dict:
    """Sizes of a step; q_lens (int32 [B]) gives per-request q lengths (varlen)."""
    lib = load()
    seq, ql = _i32(seq_lens_host), _i32(q_lens)
    z = _Sizes()
    if ql is None:
        _check(lib.okc_attn_plan_sizes(ctypes.byref(_config(cfg)), seq.ctypes.data,
                                       _options(opts), ctypes.byref(z)), "okc_attn_plan_sizes")
    else:
        _check(lib.okc_attn_plan_sizes_varlen(ctypes.byref(_config(cfg)), seq.ctypes.data, ql.ctypes.data,
                                              _options(opts), ctypes.byref(z)), "okc_attn_plan_sizes_varlen")
    return _sizes_dict(z)


def okc_attn_plan_max_sizes(cfg: dict, max_context: int, opts: dict | None = None) -> dict:
    """Bounds of okc_attn_plan_sizes over every step whose requests hold at
    most max_context tokens after it (see the header)."""
    z = _Sizes()
    _check(load().okc_attn_plan_max_sizes(ctypes.byref(_config(cfg)), max_context, _options(opts), ctypes.byref(z)),
           "okc_attn_plan_max_sizes")
    return _sizes_dict(z)


def okc_attn_plan_workspace_size(cfg: dict, max_total_ctx: int) -> int:
    n = ctypes.c_size_t(0)
    _check(load().okc_attn_plan_workspace_size(ctypes.byref(_config(cfg)), max_total_ctx, ctypes.byref(n)),
           "okc_attn_plan_workspace_size")
    return n.value


def okc_attn_plan_items(cfg: dict, seq_lens_host, opts: dict | None = None) -> np.ndarray:
    """The plan's split work list in launch order: int32 [items, 3] rows of
    (request, first key, end key) (see the header). Host only when opts give
    both ctas_per_sm and sm_count."""
    lib = load()
    seq = np.ascontiguousarray(seq_lens_host, dtype=np.int32)
    n = ctypes.c_int32(0)
    _check(lib.okc_attn_plan_items(ctypes.byref(_config(cfg)), seq.ctypes.data, _options(opts),
                                   None, 0, ctypes.byref(n)), "okc_attn_plan_items")
    out = np.zeros((n.value, 3), dtype=np.int32)
    _check(lib.okc_attn_plan_items(ctypes.byref(_config(cfg)), seq.ctypes.data, _options(opts),
                                   out.ctypes.data, n.value, ctypes.byref(n)),
           "okc_attn_plan_items")
    return out


def okc_attn_plan_items_varlen(cfg: dict, seq_lens_host, q_lens, opts: dict | None = None) -> np.ndarray:
    """The split work list of a varlen step: int32 [items, 4] rows of (request,
    first token of the item's query block, first key, end key)."""
    lib = load()
    seq, ql = _i32(seq_lens_host), _i32(q_lens)
    n = ctypes.c_int32(0)
    args = (ctypes.byref(_config(cfg)), seq.ctypes.data, _data(ql), _options(opts))
    _check(lib.okc_attn_plan_items_varlen(*args, None, 0, ctypes.byref(n)), "okc_attn_plan_items_varlen")
    out = np.zeros((n.value, 4), dtype=np.int32)
    _check(lib.okc_attn_plan_items_varlen(*args, out.ctypes.data, n.value, ctypes.byref(n)),
           "okc_attn_plan_items_varlen")
    return out


class Plan:
    """Owns an okc_attn_plan_t handle (destroyed with the object)."""

    def __init__(self, handle, cfg, workspace):
        self.handle = handle
        self.cfg = cfg  # the caller's config (not copied: plans are made every step)
        self.workspace = workspace  # keep the device buffer alive with the plan

    def update(self, seq_lens_host, stream=None, q_lens=None):
        """Re-plan in place for the next step's host lengths (see the header);
        q_lens: new per-request q lengths (varlen), else the plan keeps its own."""
        seq, ql = _i32(seq_lens_host), _i32(q_lens)
        if ql is None:
            _check(load().okc_attn_plan_update(self.handle, seq.ctypes.data, _stream(stream)),
                   "okc_attn_plan_update")
        else:
            _check(load().okc_attn_plan_update_varlen(self.handle, seq.ctypes.data, ql.ctypes.data, _stream(stream)),
                   "okc_attn_plan_update_varlen")
        return self

    @property
    def sizes(self) -> dict:
        z = _Sizes()
        _check(load().okc_attn_plan_get_sizes(self.handle, ctypes.byref(z)), "okc_attn_plan_get_sizes")
        return _sizes_dict(z)

    def scratch_sizes(self) -> dict:
        z = _Sizes()
        _check(load().okc_attn_plan_scratch_sizes(self.handle, ctypes.byref(z)), "okc_attn_plan_scratch_sizes")
        return _sizes_dict(z)

    def close(self):
        if self.handle is not None and _lib is not None:
            _lib.okc_attn_plan_destroy(self.handle)
        self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def okc_attn_plan(cfg: dict, seq_lens_host, workspace, opts: dict | None = None, stream=None,
                  q_lens=None) -> Plan:
    """The step's plan in `workspace`; q_lens (int32 [B]) makes it a varlen plan."""
    lib = load()
    seq, ql = _i32(seq_lens_host), _i32(q_lens)
    h = ctypes.c_void_p()
    nbytes = workspace.numel() * workspace.element_size()
    if ql is None:
        _check(lib.okc_attn_plan(ctypes.byref(_config(cfg)), seq.ctypes.data,
                                 _options(opts), _ptr(workspace), nbytes, _stream(stream), ctypes.byref(h)),
               "okc_attn_plan")
    else:
        _check(lib.okc_attn_plan_varlen(ctypes.byref(_config(cfg)), seq.ctypes.data, ql.ctypes.data,
                                        _options(opts), _ptr(workspace), nbytes, _stream(stream), ctypes.byref(h)),
               "okc_attn_plan_varlen")
    return Plan(h, cfg, workspace)


def okc_attn_plan_create(cfg: dict, seq_lens_host, workspace, stream=None) -> Plan:
    """okc_attn_plan with the default options."""
    seq = np.ascontiguousarray(seq_lens_host, dtype=np.int32)
    h = ctypes.c_void_p()
    nbytes = workspace.numel() * workspace.element_size()
    _check(load().okc_attn_plan_create(ctypes.byref(_config(cfg)), seq.ctypes.data,
                                       _ptr(workspace), nbytes, _stream(stream), ctypes.byref(h)),
           "okc_attn_plan_create")
    return Plan(h, cfg, workspace)


def okc_attn_plan_read_errors(plan: Plan, stream=None) -> int:
    v = ctypes.c_uint32()
    _check(load().okc_attn_plan_read_errors(plan.handle, _stream(stream), ctypes.byref(v)),
           "okc_attn_plan_read_errors")
    return v.value


def okc_attn_plan_clear_errors(plan: Plan, stream=None):
    _check(load().okc_attn_plan_clear_errors(plan.handle, _stream(stream)), "okc_attn_plan_clear_errors")


def okc_selftest_bounded_wait(err, limit_us: int, stream=None):
    """Launch the bounded-wait diagnostic (see the header); `err` is a device
    uint32 tensor that receives OKC_DEVERR_TIMEOUT when the wait gives up."""
    _check(load().okc_selftest_bounded_wait(_ptr(err), limit_us, _stream(stream)), "okc_selftest_bounded_wait")


def okc_rope_table_init(rope_theta: float, num_positions: int, table, stream=None):
    _check(load().okc_rope_table_init(rope_theta, num_positions, _ptr(table), _stream(stream)),
           "okc_rope_table_init")


def okc_prepare_qkv(plan: Plan, qkv, positions, cache_loc, k_cache, v_cache, k_scale, v_scale,
                    rope_table, q_fp8, stream=None):
    npos = 0 if rope_table is None else rope_table.shape[0]
    _check(load().okc_prepare_qkv(plan.handle, _ptr(qkv), _ptr(positions), _ptr(cache_loc),
                                  _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                  _ptr(rope_table), npos, _ptr(q_fp8), _stream(stream)),
           "okc_prepare_qkv")


def okc_attn_decode(plan: Plan, q_fp8, k_cache, v_cache, k_scale, v_scale, page_table,
                    cache_seqlens, cu_seqlens_q, seq_lens, o_partial, lse_partial, stream=None):
    _check(load().okc_attn_decode(plan.handle, _ptr(q_fp8), _ptr(k_cache), _ptr(v_cache),
                                  _ptr(k_scale), _ptr(v_scale), _ptr(page_table),
                                  _ptr(cache_seqlens), _ptr(cu_seqlens_q), _ptr(seq_lens),
                                  _ptr(o_partial), _ptr(lse_partial), _stream(stream)),
           "okc_attn_decode")


def okc_attn_combine_normgate(plan: Plan, o_partial, lse_partial, qkv, norm_weight, eps, out,
                              stream=None):
    _check(load().okc_attn_combine_normgate(plan.handle, _ptr(o_partial), _ptr(lse_partial),
                                            _ptr(qkv), _ptr(norm_weight), eps, _ptr(out),
                                            _stream(stream)),
           "okc_attn_combine_normgate")


def okc_attn_step(plan: Plan, qkv, positions, cache_loc, k_cache, v_cache, k_scale, v_scale,
                  rope_table, page_table, cache_seqlens, cu_seqlens_q, seq_lens, norm_weight, eps,
                  o_partial, lse_partial, out, stream=None):
    """The whole block in one launch (see the header)."""
    npos = 0 if rope_table is None else rope_table.shape[0]
    _check(load().okc_attn_step(plan.handle, _ptr(qkv), _ptr(positions), _ptr(cache_loc), _ptr(k_cache),
                                _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(rope_table), npos,
                                _ptr(page_table), _ptr(cache_seqlens), _ptr(cu_seqlens_q), _ptr(seq_lens),
                                _ptr(norm_weight), eps, _ptr(o_partial), _ptr(lse_partial), _ptr(out),
                                _stream(stream)),
           "okc_attn_step")


STEP_IO = ("qkv", "positions", "cache_loc", "cache_seqlens", "cu_seqlens_q", "seq_lens", "page_table", "out")


class HostStepIO:
    """The buffers of okc_attn_step_host marshalled once: host / dev map each
    name of STEP_IO to a host tensor (pinned and mapped: read in place) and
    the device buffer used when it is not. Reuse it for every step that uses
    the same buffers (it keeps the tensors alive)."""

    def __init__(self, host: dict, dev: dict):
        self.host, self.dev = dict(host), dict(dev)
        self.struct = _HostStep(
            **{k + "_host": (None if host.get(k) is None else host[k].data_ptr()) for k in STEP_IO},
            **{k: (None if dev.get(k) is None else dev[k].data_ptr()) for k in STEP_IO})
        self.ref = ctypes.byref(self.struct)


def okc_attn_step_host(plan: Plan, host, dev, k_cache, v_cache, k_scale, v_scale, rope_table,
                       norm_weight, eps, o_partial, lse_partial, stream=None):
    """One step from host buffers (see the header); returns once the output is
    in host["out"]. `host` is a HostStepIO (then `dev` is None) or the host
    dict of one, with `dev` its device dict."""
    io = host if isinstance(host, HostStepIO) else HostStepIO(host, dev)
    npos = 0 if rope_table is None else rope_table.shape[0]
    _check(load().okc_attn_step_host(plan.handle, io.ref, _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
                                     _ptr(v_scale), _ptr(rope_table), npos, _ptr(norm_weight), eps,
                                     _ptr(o_partial), _ptr(lse_partial), _stream(stream)),
           "okc_attn_step_host")


def okc_attn_decode_combine_noalloc(cfg: dict, seq_lens_host, q_fp8, k_cache, v_cache, k_scale,
                                    v_scale, page_table, cache_seqlens, cu_seqlens_q, seq_lens, qkv,
                                    norm_weight, eps, out, stream=None):
    """Decode + merge + norm-gate without any caller-provided scratch, for
    callers that cannot allocate device memory (see the header)."""
    seq = np.ascontiguousarray(seq_lens_host, dtype=np.int32)
    _check(load().okc_attn_decode_combine_noalloc(
        ctypes.byref(_config(cfg)), seq.ctypes.data, _ptr(q_fp8), _ptr(k_cache),
        _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(page_table), _ptr(cache_seqlens),
        _ptr(cu_seqlens_q), _ptr(seq_lens), _ptr(qkv), _ptr(norm_weight), eps, _ptr(out),
        _stream(stream)), "okc_attn_decode_combine_noalloc")


class AttnStep:
    """One step of the block on device tensors: makes the plan, owns the
    workspace and scratch (allocated once through torch), and issues the three
    entry points on a stream.

    inputs: dict of device tensors named as in the problem file's `Inputs`
    (qkv bf16 [T, 2304], positions, cache_loc, cache_seqlens, cu_seqlens_q,
    seq_lens, page_table, k_cache, v_cache (uint8 views), k_scale, v_scale) plus
    norm_weight (bf16 [64] or None) and rope_table (float32 or None).
    """

    def __init__(self, cfg: dict, seq_lens_host, device=None, opts: dict | None = None, stream=None,
                 q_lens=None):
        import torch
        self.cfg = dict(cfg)
        self.device = device or torch.device("cuda")
        sizes = okc_attn_plan_sizes(cfg, seq_lens_host, opts, q_lens)
        self.workspace = torch.empty(sizes["workspace_bytes"], dtype=torch.uint8, device=self.device)
        self.plan = okc_attn_plan(cfg, seq_lens_host, self.workspace, opts, stream, q_lens)
        sizes = self.plan.sizes
        self.sizes = sizes
        # a fixed-capacity plan's scratch serves every step within its max_context
        scratch = okc_attn_plan_max_sizes(cfg, opts["max_context"], opts) if (opts or {}).get("max_context") else sizes
        self.q_fp8 = torch.empty(sizes["q_fp8_bytes"], dtype=torch.uint8, device=self.device)
        self.o_partial = torch.empty(max(16, scratch["o_partial_bytes"]) // 4, dtype=torch.float32, device=self.device)
        self.lse_partial = torch.empty(max(16, scratch["lse_partial_bytes"]) // 4, dtype=torch.float32,
                                       device=self.device)
        T = sizes["num_tokens"]
        self.out = torch.empty((T, cfg["num_q_heads"] * cfg["head_dim"]), dtype=torch.bfloat16, device=self.device)

    def run(self, inp: dict, eps: float = 1e-5, out=None, stream=None):
        out = self.out if out is None else out
        okc_prepare_qkv(self.plan, inp["qkv"], inp["positions"], inp["cache_loc"], inp["k_cache"],
                        inp["v_cache"], inp["k_scale"], inp["v_scale"], inp.get("rope_table"),
                        self.q_fp8, stream)
        okc_attn_decode(self.plan, self.q_fp8, inp["k_cache"], inp["v_cache"], inp["k_scale"],
                        inp["v_scale"], inp["page_table"], inp["cache_seqlens"], inp["cu_seqlens_q"],
                        inp.get("seq_lens"), self.o_partial, self.lse_partial, stream)
        okc_attn_combine_normgate(self.plan, self.o_partial, self.lse_partial, inp["qkv"],
                                  inp.get("norm_weight"), eps, out, stream)
        return out

    def run_fused(self, inp: dict, eps: float = 1e-5, out=None, stream=None):
        """The same step through okc_attn_step (one launch)."""
        out = self.out if out is None else out
        okc_attn_step(self.plan, inp["qkv"], inp["positions"], inp["cache_loc"], inp["k_cache"],
                      inp["v_cache"], inp["k_scale"], inp["v_scale"], inp.get("rope_table"),
                      inp["page_table"], inp["cache_seqlens"], inp["cu_seqlens_q"], inp.get("seq_lens"),
                      inp.get("norm_weight"), eps, self.o_partial, self.lse_partial, out, stream)
        return out

    def errors(self, stream=None) -> int:
        return okc_attn_plan_read_errors(self.plan, stream)
