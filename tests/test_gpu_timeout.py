"""The kernels' bounded-wait failure path, exercised without a fault: a wait
on an mbarrier that nothing arrives on gives up after its limit, sets
PA_STATUS_TIMEOUT and returns, and the CUDA context stays usable (the pages'
only device failure mode is a timeout: pypto-serving top-k PR, "Exactness
Design").  No bulk copy is in flight and nothing faults or hangs: the wait is
bounded by construction (limit in wall-clock time and in polls)."""
import time

import pytest
import torch

import workloads as W
from pa_testutil import ATOL, assert_close, oracle_decode

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("limit_us", [1, 2000, 20000])
def test_wait_gives_up_and_reports_timeout(cuda_lib, limit_us):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    cuda_lib.pa_wait_selftest(limit_us, status=st)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    # exactly the timeout bit: no wait claimed a phase nobody completed
    assert int(st.item()) == cuda_lib.PA_STATUS_TIMEOUT
    # gave up near its limit (one sleep slice per poll, checked every 16 polls)
    assert dt < limit_us * 1e-6 + 0.5, dt


def test_context_usable_after_a_timeout(cuda_lib):
    st = cuda_lib.pa_wait_selftest(1000)
    case = W.tiny_decode()
    c = case.to("cuda")
    out = cuda_lib.pa_decode(c.q, c.k_cache, c.v_cache, c.block_table, c.context_lens, c.scale,
                             out_dtype=torch.float32, num_splits=2)
    torch.cuda.synchronize()
    assert int(st.item()) == cuda_lib.PA_STATUS_TIMEOUT
    assert_close(out, oracle_decode(case), atol=ATOL, what="decode after a timeout")
