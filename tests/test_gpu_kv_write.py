"""pa_kv_write on the GPU against the oracle's byte copy: bit-exact, no stray
writes, invalid sequences skipped and flagged."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from pa_testutil import cache_bits, dev_status

pytestmark = pytest.mark.gpu


def _check_write(pa, case):
    c = case.to("cuda")
    st = dev_status()
    pa.pa_kv_write(c.k_new, c.v_new, c.k_cache, c.v_cache, c.block_table, c.context_lens,
                   c.chunk_lens, status=st)
    torch.cuda.synchronize()
    kc, vc, skipped = oracle.kv_write(case.k_new, case.v_new, case.k_cache, case.v_cache,
                                      case.block_table, case.context_lens, case.chunk_lens,
                                      case.num_pages, case.max_pages_per_seq)
    assert np.array_equal(cache_bits(c.k_cache), kc)
    assert np.array_equal(cache_bits(c.v_cache), vc)
    return int(st.item()), skipped


def test_decode_write_tiny(cuda_lib):
    st, sk = _check_write(cuda_lib, W.tiny_decode(with_new=True))
    assert st == 0 and sk == 0


def test_decode_write_qwen3_32b_ragged(cuda_lib):
    st, sk = _check_write(cuda_lib, W.qwen3_32b_ragged())
    assert st == 0 and sk == 0


def test_prefill_write_4096_tokens(cuda_lib):
    st, sk = _check_write(cuda_lib, W.chunked_prefill())
    assert st == 0 and sk == 0


@pytest.mark.parametrize("ctx,chunk", [([1, 128, 129, 300], [1, 128, 2, 171]),
                                       ([5, 0, 257], [5, 0, 1])])
def test_ragged_chunks(cuda_lib, ctx, chunk):
    case = W.custom_case(300 + sum(chunk), ctx, Hq=4, Hkv=2, chunk_lens=chunk, with_new=True)
    st, sk = _check_write(cuda_lib, case)
    assert st == 0 and sk == 0


def test_wide_kv_heads(cuda_lib):
    case = W.custom_case(310, [200, 3], Hq=16, Hkv=16, chunk_lens=[7, 3], with_new=True)
    st, sk = _check_write(cuda_lib, case)
    assert st == 0 and sk == 0


def test_invalid_page_skips_sequence_and_flags(cuda_lib):
    case = W.custom_case(311, [10, 300], Hq=4, Hkv=2, chunk_lens=[2, 4], with_new=True)
    case.block_table[1, 0] = case.num_pages + 5          # prior page out of range
    st, sk = _check_write(cuda_lib, case)
    assert sk == 1 and st & cuda_lib.PA_STATUS_BAD_PAGE


def test_bad_lengths_flag(cuda_lib):
    case = W.custom_case(312, [10, 20], Hq=4, Hkv=2, chunk_lens=[2, 4], with_new=True)
    case.chunk_lens[0] = 11                               # more new tokens than context
    case.k_new = torch.cat([case.k_new, case.k_new, case.k_new[:3]])   # 15 rows = sum
    case.v_new = torch.cat([case.v_new, case.v_new, case.v_new[:3]])
    st, sk = _check_write(cuda_lib, case)
    assert sk == 1 and st & cuda_lib.PA_STATUS_BAD_LENGTH


def test_token_count_mismatch_flags(cuda_lib):
    case = W.custom_case(313, [10, 20], Hq=4, Hkv=2, chunk_lens=[2, 4], with_new=True).to("cuda")
    st = dev_status()
    cuda_lib.pa_kv_write(case.k_new[:5], case.v_new[:5], case.k_cache, case.v_cache,
                         case.block_table, case.context_lens, case.chunk_lens, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & cuda_lib.PA_STATUS_BAD_TOKENS
