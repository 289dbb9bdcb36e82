"""pa_combine on the GPU against the oracle's log-sum-exp merge."""
import numpy as np
import pytest
import torch

import oracle
from pa_testutil import assert_close, assert_close_bf16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,Hq,S", [(1, 1, 1), (3, 8, 4), (16, 40, 7), (2, 5, 33)])
def test_combine_matches_oracle(cuda_lib, B, Hq, S):
    g = torch.Generator().manual_seed(B * 100 + S)
    po = torch.randn(B, Hq, S, 128, generator=g)
    pl = torch.randn(B, Hq, S, generator=g) * 4
    if S > 1:
        pl[0, 0, 0] = -float("inf")                    # an empty state
        po[0, 0, 0] = float("nan")                     # never read
    ref = oracle.combine(po.double().numpy().reshape(B * Hq, S, 128),
                         pl.double().numpy().reshape(B * Hq, S)).reshape(B, Hq, 128)
    out = cuda_lib.pa_combine(po.cuda(), pl.cuda(), out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert_close(out, ref, atol=1e-5, what="combine f32")
    outb = cuda_lib.pa_combine(po.cuda(), pl.cuda(), out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert_close_bf16(outb, ref, what="combine bf16")


def test_all_empty_and_invalid_rows_are_zero(cuda_lib):
    po = torch.randn(1, 3, 4, 128)
    pl = torch.randn(1, 3, 4)
    pl[0, 0] = -float("inf")
    pl[0, 1, 2] = float("inf")
    out = cuda_lib.pa_combine(po.cuda(), pl.cuda(), out_dtype=torch.float32).cpu()
    assert torch.count_nonzero(out[0, 0]) == 0 and torch.count_nonzero(out[0, 1]) == 0
    assert torch.count_nonzero(out[0, 2]) > 0
