"""The kernels' bounded waits give up without faulting or hanging: the
bounded-wait diagnostic waits on an mbarrier that nothing arrives on, with the
same wait the kernels use, flags OKC_DEVERR_TIMEOUT once its limit has passed,
and returns; the context then still runs the block and matches the oracle."""
import pytest
import torch

import workloads as W
from parity_util import full_check

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("limit_us", [500, 5000])
def test_bounded_wait_gives_up_and_the_context_stays_usable(cuda_lib, limit_us):
    okc = cuda_lib
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    okc.okc_selftest_bounded_wait(err, limit_us, s)
    e1.record(s)
    torch.cuda.synchronize()
    assert int(err.item()) & okc.DEVERR_TIMEOUT
    ms = e0.elapsed_time(e1)
    assert limit_us / 1000.0 <= ms < 1000.0, ms  # gave up after its limit, well before the kernels' 1 s
    cfg = W.config("sliding_decode", batch=4, seq=("uniform", 500, 3000))
    full_check(cfg, W.generate(cfg))
