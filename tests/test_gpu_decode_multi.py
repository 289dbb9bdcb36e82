"""pa_decode_multi (q_len new tokens per sequence on the decode kernel) on the
GPU against the FP64 oracle's causal attention with chunk_lens = q_len."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from pa_testutil import assert_close, dev_status, oracle_prefill, sample_rows

pytestmark = pytest.mark.gpu

BAL = -1  # PA_SPLITS_BALANCED


def _write(pa, c):
    st = dev_status()
    pa.pa_kv_write(c.k_new, c.v_new, c.k_cache, c.v_cache, c.block_table, c.context_lens,
                   c.chunk_lens, status=st)
    return st


def _oracle_after_write(case, rows=None):
    kc, vc, _ = oracle.kv_write(case.k_new, case.v_new, case.k_cache, case.v_cache,
                                case.block_table, case.context_lens, case.chunk_lens,
                                case.num_pages, case.max_pages_per_seq)
    return oracle.attention(case.q, kc, vc, case.block_table, case.context_lens,
                            case.chunk_lens, case.scale, case.Hq, case.Hkv, case.num_pages,
                            case.max_pages_per_seq, rows=rows)


@pytest.mark.parametrize("q_len", [1, 2, 3, 4, 8, 16])
@pytest.mark.parametrize("splits", [0, 1, 3, BAL])
def test_ragged_batch_all_rows(cuda_lib, q_len, splits):
    """Contexts that put the new tokens inside one page, across a page boundary,
    at the very start of the cache and at a page's end."""
    ctx = [q_len, 130, 127 + q_len, 1000, 129, 256 + q_len // 2]
    case = W.custom_case(700 + q_len, ctx, Hq=8, Hkv=2, chunk_lens=[q_len] * len(ctx),
                         with_new=True)
    c = case.to("cuda")
    st = _write(cuda_lib, c)
    out = cuda_lib.pa_decode_multi(c.q, c.k_cache, c.v_cache, c.block_table, c.context_lens,
                                   q_len, c.scale, out_dtype=torch.float32, num_splits=splits,
                                   status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert_close(out, _oracle_after_write(case), what=f"q_len={q_len} splits={splits}")


@pytest.mark.parametrize("Hq,Hkv,q_len", [(40, 8, 4), (64, 8, 2), (16, 1, 3), (32, 2, 5), (40, 8, 7)])
def test_head_layouts(cuda_lib, Hq, Hkv, q_len):
    """G query heads per KV head: items of up to 32 (token, head) columns; 40/8
    with q_len 7 takes one 20-column and one 15-column token group."""
    ctx = [700, 129, 2000]
    case = W.custom_case(720 + Hq, ctx, Hq=Hq, Hkv=Hkv, chunk_lens=[q_len] * 3, with_new=True)
    c = case.to("cuda")
    st = _write(cuda_lib, c)
    out = cuda_lib.pa_decode_multi(c.q, c.k_cache, c.v_cache, c.block_table, c.context_lens,
                                   q_len, c.scale, out_dtype=torch.float32, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert_close(out, _oracle_after_write(case), what=f"Hq={Hq} Hkv={Hkv} q_len={q_len}")


def test_agrees_with_prefill_kernel(cuda_lib):
    """The same step through pa_prefill_chunk (chunk_lens = q_len): both kernels
    meet the oracle, and each other within twice its tolerance."""
    q_len = 4
    case = W.custom_case(740, [300, 1500, 4], Hq=40, Hkv=8, chunk_lens=[q_len] * 3,
                         with_new=True)
    c = case.to("cuda")
    st = _write(cuda_lib, c)
    a = cuda_lib.pa_decode_multi(c.q, c.k_cache, c.v_cache, c.block_table, c.context_lens,
                                 q_len, c.scale, out_dtype=torch.float32, status=st)
    b = cuda_lib.pa_prefill_chunk(c.q, c.k_cache, c.v_cache, c.block_table, c.context_lens,
                                  c.chunk_lens, c.scale, out_dtype=torch.float32, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = _oracle_after_write(case)
    assert_close(a, ref, what="decode_multi")
    assert_close(b, ref, what="prefill_chunk")


@pytest.mark.parametrize("splits", [0, 1, 4, BAL])
def test_q_len_one_is_decode_bitwise(cuda_lib, splits):
    case = W.qwen3_14b_decode_b16().to("cuda")
    a = cuda_lib.pa_decode(case.q, case.k_cache, case.v_cache, case.block_table,
                           case.context_lens, case.scale, out_dtype=torch.float32,
                           num_splits=splits)
    b = cuda_lib.pa_decode_multi(case.q, case.k_cache, case.v_cache, case.block_table,
                                 case.context_lens, 1, case.scale, out_dtype=torch.float32,
                                 num_splits=splits)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("splits", [1, 2, BAL])
def test_short_and_empty_sequences(cuda_lib, splits):
    """0 < context < q_len makes the sequence invalid (flag, zero rows); context 0
    gives zero rows without a flag; the other sequences are unaffected."""
    q_len = 4
    ctx = [600, 300, 900]
    case = W.custom_case(760, ctx, Hq=8, Hkv=2, chunk_lens=[q_len] * 3, with_new=True)
    c = case.to("cuda")
    st = _write(cuda_lib, c)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = _oracle_after_write(case).reshape(3, q_len, 8, 128)
    for lens, bad in (([600, 3, 900], cuda_lib.PA_STATUS_BAD_LENGTH), ([600, 0, 900], 0)):
        st2 = dev_status()
        cl = torch.tensor(lens, dtype=torch.int32, device="cuda")
        out = cuda_lib.pa_decode_multi(c.q, c.k_cache, c.v_cache, c.block_table, cl, q_len,
                                       c.scale, out_dtype=torch.float32, num_splits=splits,
                                       status=st2)
        torch.cuda.synchronize()
        assert int(st2.item()) == bad
        o = out.reshape(3, q_len, 8, 128)
        assert torch.count_nonzero(o[1]).item() == 0
        assert_close(o[0], ref[0], what=f"seq 0 beside {lens}")
        assert_close(o[2], ref[2], what=f"seq 2 beside {lens}")


def test_full_size_sampled(cuda_lib):
    """64 sequences x 4096 tokens, q_len 4, 40/8 heads: the launch the benchmark
    times, checked on sampled rows (every new-token position among them)."""
    case = W.multi_token_decode()
    c = case.to("cuda")
    st = _write(cuda_lib, c)
    out = cuda_lib.pa_decode_multi(c.q, c.k_cache, c.v_cache, c.block_table, c.context_lens,
                                   4, c.scale, out_dtype=torch.float32, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    T = case.T
    rows = sample_rows(T, 40, 96, seed=3, extra=[j * 40 + 7 for j in range(4)] +
                       [(T - 4 + j) * 40 + 39 for j in range(4)])
    ref = _oracle_after_write(case, rows=rows)
    got = out.reshape(-1, 128)[torch.as_tensor(rows, device="cuda")]
    assert_close(got, ref, what="multi-token b64 q4 sampled")
