"""No stray reads: with every cache row that no query of the step may read set
to an E4M3 NaN (tests/poison.py: unused pages, positions past each request's
last key, positions before its window's first 8-row group), each decode path
still matches the oracle (a NaN read would reach the output even at P = 0),
leaves the poisoned rows as they were, and flags nothing."""
import pytest

import workloads as W
from parity_util import full_check
from poison import poison

pytestmark = pytest.mark.gpu

CASES = [
    ("sliding_decode", dict(batch=6, seq=("uniform", 500, 5000)), None),
    ("sliding_decode", dict(batch=6, seq=("uniform", 500, 5000)), {"chunk_keys": 100}),
    ("verify_block", dict(batch=4, seq=("uniform", 2000, 5000)), None),             # tcgen05, TMA tiles
    ("verify_block", dict(batch=4, seq=("uniform", 2000, 5000)), {"chunk_keys": 200}),
    ("verify_block", dict(batch=4, seq=("uniform", 2000, 5000), page_size=1), None),  # tcgen05, cp.async
    ("verify_block", dict(batch=4, seq=("uniform", 2000, 5000)), {"flags": 2}),     # warp-level MMA decode
    ("mixed_full_decode", dict(batch=12, seq=("loguniform", 1, 20000)), None),
    ("full_decode_32k", dict(batch=2, seq=("const", 3000), page_size=16), None),
]


@pytest.mark.parametrize("name,over,opts", CASES)
def test_no_decode_path_reads_a_row_no_query_may_see(cuda_lib, name, over, opts):
    cfg = W.config(name, **over)
    inp = W.generate(cfg)
    pcfg, bad = poison(cfg, inp)
    full_check(pcfg, bad, opts=opts)
    full_check(pcfg, bad, opts=opts, fused=True)  # one kernel where the step has that form
