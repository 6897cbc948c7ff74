"""The oracle reads only what each query may see: with every cache row outside
a request's readable positions set to an E4M3 NaN (tests/poison.py), the
oracle's step is bit-identical to the step on the unpoisoned caches (q codes,
written rows, attention output, block output), for window and full layers,
decode and verify blocks, 1-row and 64-row pages."""
import numpy as np
import pytest

import oracle
import workloads as W
from poison import poison

CASES = {
    "tiny_sliding_decode": {},
    "sliding_decode": dict(batch=4, seq=("uniform", 500, 3000)),
    "verify_block": dict(batch=3, seq=("uniform", 2000, 4000)),
    "mixed_full_decode": dict(batch=6, seq=("loguniform", 1, 3000)),
    "full_decode_32k": dict(batch=2, seq=("const", 900)),
}


@pytest.mark.parametrize("name", list(CASES))
def test_oracle_ignores_rows_no_query_may_read(name):
    cfg = W.config(name, **CASES[name])
    inp = W.generate(cfg)
    pcfg, bad = poison(cfg, inp)
    assert bad["poisoned_rows"] >= 3 * cfg["page_size"]
    a, b = oracle.step(cfg, inp), oracle.step(pcfg, bad)
    for k in ("q8", "out"):
        assert np.array_equal(a[k], b[k]), k
    assert np.array_equal(a["o"], b["o"])  # fp64 attention, bit for bit
    assert np.all(np.isfinite(b["o"]))
    loc = inp["cache_loc"]
    for k in ("k_cache", "v_cache"):
        assert np.array_equal(a[k].reshape(-1, 128)[loc], b[k].reshape(-1, 128)[loc]), k
        assert np.all(b[k].reshape(-1, 128)[-3 * cfg["page_size"]:] == 0x7F)  # unused pages untouched
