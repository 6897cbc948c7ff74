"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times (okc_attn_step with the default plan, in the form the plan
chooses) and through the three calls: every written cache row is compared
(and every q byte on the three-call path); the bf16 output is compared on
sampled query rows that the oracle computes one by one (all rows where that is
cheap)."""
import numpy as np
import pytest

import workloads as W
from parity_util import full_check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib):
    return cuda_lib


def _rows_mask(cfg, inp, n_requests, seed):
    """All query rows of a sample of requests (always including the longest)."""
    B, L = cfg["batch"], cfg["q_len"]
    rng = np.random.default_rng(seed)
    pick = set(rng.choice(B, size=min(B, n_requests), replace=False).tolist())
    pick.add(int(np.argmax(inp["seq_lens"])))
    pick.add(int(np.argmin(inp["seq_lens"])))
    mask = np.zeros((B * L, 16), np.uint8)
    for b in pick:
        mask[b * L:(b + 1) * L] = 1
    return mask


@pytest.mark.parametrize("name,n_req", [
    ("sliding_decode", None),
    ("full_decode_32k", 6),
    ("verify_block", None),
    ("mixed_full_decode", 24),
])
def test_full_size(name, n_req):
    cfg = W.config(name)
    inp = W.generate(cfg)
    mask = None if n_req is None else _rows_mask(cfg, inp, n_req, seed=cfg["seed"])
    rep = full_check(cfg, inp, rows_mask=mask, fused=True, plan_form=True)  # as the benchmark runs it
    print(name, "step", rep)
    rep = full_check(cfg, inp, rows_mask=mask)
    print(name, "three calls", rep)
