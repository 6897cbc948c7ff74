"""CPU oracle of the paged-FP8 gated attention block.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may use it; the CUDA library never does, and this
module imports nothing from it.

A thin numpy/ctypes driver over ``okc_oracle.c`` (plain C, compiled with gcc,
``-ffp-contract=off``). Every step follows "012-attention-local-splits.py"
(the SGLang Muse Spark attention problem file) literally; see the C source for
the citation of each function and the readings taken where the page is silent.

Arrays: bf16 values are ``uint16`` bit patterns, E4M3 values ``uint8`` codes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "okc_oracle.c")
_LIB_DIR = os.path.join(_HERE, "lib")
_LIB = os.path.join(_LIB_DIR, "libokc_oracle.so")
_lock = threading.Lock()
_lib = None

HEAD_DIM = 64


def build(force: bool = False) -> str:
    """Compile the oracle into oracle/lib/libokc_oracle.so (gcc, plain -O2)."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


class _Cfg(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("batch", "q_len", "hq", "hkv", "page_size", "window", "max_pages", "num_pages")] + \
               [(n, ctypes.c_float) for n in ("rope_theta", "qk_scale_factor", "sm_scale", "kv_scale")] + \
               [("q_norm", ctypes.c_int32)]


def _bind(lib):
    P = ctypes.c_void_p
    i64 = ctypes.c_int64
    lib.orc_bf16_round.restype = ctypes.c_double
    lib.orc_bf16_round.argtypes = [ctypes.c_double]
    lib.orc_bf16_round_array.argtypes = [P, P, i64]
    lib.orc_e4m3_code_array.argtypes = [P, P, i64]
    lib.orc_e4m3_value_array.argtypes = [P, P, i64]
    lib.orc_rope_inv_freq.argtypes = [ctypes.c_float, P]
    lib.orc_rope_row.argtypes = [ctypes.c_float, i64, P, P]
    lib.orc_prepare.restype = i64
    lib.orc_prepare.argtypes = [ctypes.POINTER(_Cfg), i64, P, P, P, P, P,
                                ctypes.c_float, ctypes.c_float, P]
    lib.orc_attention.restype = i64
    lib.orc_attention.argtypes = [ctypes.POINTER(_Cfg), P, P, P, ctypes.c_float,
                                  ctypes.c_float, P, P, P, P, P, P]
    lib.orc_normgate.argtypes = [ctypes.POINTER(_Cfg), i64, P, P, P, ctypes.c_float, P, P]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


class use_library:
    """Context manager: run the oracle functions on another build of okc_oracle.c
    (the pin tests use it to show that a planted mistake fails a pin)."""

    def __init__(self, path: str):
        self.path = path

    def __enter__(self):
        global _lib
        _load()
        self.saved = _lib
        _lib = _bind(ctypes.CDLL(self.path))
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self.saved
        return False


def compile_source(src_text: str, out_path: str) -> str:
    """Compile a variant of the oracle's C source (same flags as build())."""
    c_path = out_path + ".c"
    with open(c_path, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
                    "-fno-fast-math", "-o", out_path, c_path, "-lm"], check=True)
    return out_path


def source() -> str:
    with open(_SRC) as f:
        return f.read()


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _cfg(cfg: dict) -> _Cfg:
    return _Cfg(cfg["batch"], cfg["q_len"], cfg["num_q_heads"], cfg["num_kv_heads"],
                cfg["page_size"], cfg["window"], cfg["max_pages"], cfg["num_pages"],
                cfg["rope_theta"], cfg["qk_scale_factor"], cfg["sm_scale"], cfg["kv_scale"],
                int(cfg.get("q_norm", 0)))


# ------------------------------------------------------------------ formats

def bf16_bits(x) -> np.ndarray:
    """float -> bf16 (round to nearest even), as uint16 bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, np.uint16)
    _load().orc_bf16_round_array(_ptr(x), _ptr(out), x.size)
    return out


def bf16_value(bits) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    with np.errstate(invalid="ignore"):
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def e4m3_code(x) -> np.ndarray:
    """float -> E4M3 code (round to nearest even, satfinite)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, np.uint8)
    _load().orc_e4m3_code_array(_ptr(x), _ptr(out), x.size)
    return out


def e4m3_value(codes) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(codes.shape, np.float64)
    _load().orc_e4m3_value_array(_ptr(codes), _ptr(out), codes.size)
    return out


# --------------------------------------------------------------------- RoPE

def rope_inv_freq(theta: float) -> np.ndarray:
    out = np.empty(HEAD_DIM // 2, np.float32)
    _load().orc_rope_inv_freq(ctypes.c_float(theta), _ptr(out))
    return out


def rope_row(theta: float, pos: int):
    c = np.empty(HEAD_DIM // 2, np.float32)
    s = np.empty(HEAD_DIM // 2, np.float32)
    _load().orc_rope_row(ctypes.c_float(theta), int(pos), _ptr(c), _ptr(s))
    return c, s


# -------------------------------------------------------------------- steps

def prepare(cfg: dict, inp: dict, k_cache: np.ndarray, v_cache: np.ndarray):
    """Steps 1-3. Writes k_cache / v_cache in place; returns (q8 [T,Hq,64], skipped rows)."""
    T = inp["qkv"].shape[0]
    q8 = np.zeros((T, cfg["num_q_heads"], HEAD_DIM), np.uint8)
    assert k_cache.dtype == np.uint8 and v_cache.dtype == np.uint8
    skipped = _load().orc_prepare(
        ctypes.byref(_cfg(cfg)), T, _ptr(np.ascontiguousarray(inp["qkv"], np.uint16)),
        _ptr(np.ascontiguousarray(inp["positions"], np.int64)),
        _ptr(np.ascontiguousarray(inp["cache_loc"], np.int64)), _ptr(k_cache), _ptr(v_cache),
        ctypes.c_float(float(inp["k_scale"])), ctypes.c_float(float(inp["v_scale"])), _ptr(q8))
    return q8, skipped


def attention(cfg: dict, inp: dict, q8: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
              rows_mask: np.ndarray | None = None, want_lse: bool = False):
    """Step 4 in double precision. rows_mask: uint8 [T, Hq] selecting rows to compute."""
    T = q8.shape[0]
    hq = cfg["num_q_heads"]
    o = np.zeros((T, hq, HEAD_DIM), np.float64)
    lse = np.full((T, hq), np.nan, np.float64) if want_lse else None
    mask = None if rows_mask is None else np.ascontiguousarray(rows_mask, np.uint8)
    bad = _load().orc_attention(
        ctypes.byref(_cfg(cfg)), _ptr(np.ascontiguousarray(q8)), _ptr(k_cache), _ptr(v_cache),
        ctypes.c_float(float(inp["k_scale"])), ctypes.c_float(float(inp["v_scale"])),
        _ptr(np.ascontiguousarray(inp["page_table"], np.int32)),
        _ptr(np.ascontiguousarray(inp["cache_seqlens"], np.int32)),
        _ptr(np.ascontiguousarray(inp["cu_seqlens_q"], np.int32)), _ptr(mask), _ptr(o), _ptr(lse))
    return (o, lse, bad) if want_lse else (o, bad)


def normgate(cfg: dict, o: np.ndarray, qkv: np.ndarray, weight: np.ndarray | None, eps: float,
             rows_mask: np.ndarray | None = None) -> np.ndarray:
    """Step 5: bf16 [T, Hq*64] (uint16 bits)."""
    T = o.shape[0]
    out = np.zeros((T, cfg["num_q_heads"] * HEAD_DIM), np.uint16)
    mask = None if rows_mask is None else np.ascontiguousarray(rows_mask, np.uint8)
    w = None if weight is None else np.ascontiguousarray(weight, np.uint16)
    _load().orc_normgate(ctypes.byref(_cfg(cfg)), T, _ptr(np.ascontiguousarray(o, np.float64)),
                         _ptr(np.ascontiguousarray(qkv, np.uint16)), _ptr(w), ctypes.c_float(eps),
                         _ptr(mask), _ptr(out))
    return out


def step(cfg: dict, inp: dict, rows_mask: np.ndarray | None = None) -> dict:
    """The whole block on copies of the caches: returns q8, caches, o, out."""
    k_cache = inp["k_cache"].copy()
    v_cache = inp["v_cache"].copy()
    q8, skipped = prepare(cfg, inp, k_cache, v_cache)
    o, bad = attention(cfg, inp, q8, k_cache, v_cache, rows_mask)
    out = normgate(cfg, o, inp["qkv"], inp.get("norm_weight"), inp["eps"], rows_mask)
    return {"q8": q8, "k_cache": k_cache, "v_cache": v_cache, "o": o, "out": out,
            "skipped_rows": skipped, "bad_keys": bad}
