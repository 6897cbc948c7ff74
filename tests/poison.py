"""Poisoned caches: every cache row that no query of the step may read is set
to 0x7F in both caches (an E4M3 NaN), so that a stray read shows up as a NaN
in the output. A row may be read when it holds a position of its request in
[lo & ~7, seq + L): the visible keys [lo, seq + L), lo = max(0, seq - window + 1)
on window layers (else 0), plus the up to 7 earlier positions that share the
first visible key's 8-row group (a tile of the TMA-fed verify decode starts
there and masks them). Rows of pages no request uses (extra_pages of them are
appended to the pool), positions past seq + L in a request's last page, and
positions before lo & ~7 are poisoned."""
import numpy as np


def poison(cfg: dict, inp: dict, extra_pages: int = 3):
    """Returns (cfg, inputs) with the pool grown by extra_pages and poisoned."""
    B, L, P, w = cfg["batch"], cfg["q_len"], cfg["page_size"], cfg["window"]
    cfg = dict(cfg, num_pages=cfg["num_pages"] + extra_pages)
    rows = cfg["num_pages"] * P
    keep = np.zeros(rows, bool)
    pt = inp["page_table"]
    for b in range(B):
        seq = int(inp["seq_lens"][b])
        n = seq + L
        lo = max(0, seq - w + 1) if w > 0 else 0
        pos = np.arange(lo & ~7, n)
        keep[pt[b, pos // P].astype(np.int64) * P + pos % P] = True
    out = dict(inp)
    for name in ("k_cache", "v_cache"):
        c = np.concatenate([inp[name].reshape(-1, 128), np.zeros((extra_pages * P, 128), np.uint8)])
        c[~keep] = 0x7F
        out[name] = c.reshape((cfg["num_pages"],) + inp[name].shape[1:])
    out["poisoned_rows"] = int((~keep).sum())
    return cfg, out
