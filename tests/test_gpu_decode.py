"""pa_decode (+ the combine kernel) on the GPU against the FP64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from pa_testutil import (assert_close, assert_close_bf16, cache_bits, dev_status,
                         oracle_decode, sample_rows)

pytestmark = pytest.mark.gpu


def _decode(pa, c, num_splits=0, out_dtype=torch.float32):
    st = dev_status()
    out = pa.pa_decode(c.q, c.k_cache, c.v_cache, c.block_table, c.context_lens, c.scale,
                       out_dtype=out_dtype, num_splits=num_splits, status=st)
    torch.cuda.synchronize()
    return out, int(st.item())


BAL = -1  # PA_SPLITS_BALANCED: the page-balanced schedule


@pytest.mark.parametrize("splits", [0, 1, 2, BAL])
def test_tiny(cuda_lib, splits):
    case = W.tiny_decode()
    out, st = _decode(cuda_lib, case.to("cuda"), splits)
    assert st == 0
    assert_close(out, oracle_decode(case), what="tiny")


def test_tiny_single_token_is_v_exactly(cuda_lib):
    case = W.tiny_decode()
    out, _ = _decode(cuda_lib, case.to("cuda"))
    page = int(case.block_table[0, 0])
    for g in range(8):
        v = case.v_cache[page, 0, g // 4].float()
        assert torch.equal(out[0, g].cpu(), v)


@pytest.mark.parametrize("splits", [0, 1, 3, 32, BAL])
def test_qwen3_14b_b16(cuda_lib, splits):
    case = W.qwen3_14b_decode_b16()
    out, st = _decode(cuda_lib, case.to("cuda"), splits)
    assert st == 0
    assert_close(out, oracle_decode(case), what=f"b16 splits={splits}")


def test_qwen3_14b_b16_bf16_out(cuda_lib):
    case = W.qwen3_14b_decode_b16()
    out, st = _decode(cuda_lib, case.to("cuda"), 0, torch.bfloat16)
    assert st == 0
    assert_close_bf16(out, oracle_decode(case), what="b16 bf16")


def test_qwen3_14b_b128_full_size_sampled(cuda_lib):
    """The bandwidth-bound workload at full size, in the launch configuration the
    benchmark times (automatic splits), checked on sampled rows."""
    case = W.qwen3_14b_decode_b128()
    out, st = _decode(cuda_lib, case.to("cuda"), 0)
    assert st == 0
    rows = sample_rows(128, 40, 96, seed=1, extra=[39, 40, 41, 5119 - 40])
    ref = oracle_decode(case, rows=rows)
    got = out.reshape(-1, 128)[torch.as_tensor(rows, device="cuda")]
    assert_close(got, ref, what="b128 sampled")


def test_qwen3_32b_ragged_with_write(cuda_lib):
    case = W.qwen3_32b_ragged()
    c = case.to("cuda")
    st = dev_status()
    cuda_lib.pa_kv_write(c.k_new, c.v_new, c.k_cache, c.v_cache, c.block_table, c.context_lens,
                         None, status=st)
    out = cuda_lib.pa_decode(c.q, c.k_cache, c.v_cache, c.block_table, c.context_lens, c.scale,
                             out_dtype=torch.float32, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    kc, vc, _ = oracle.kv_write(case.k_new, case.v_new, case.k_cache, case.v_cache,
                                case.block_table, case.context_lens, None, case.num_pages,
                                case.max_pages_per_seq)
    assert np.array_equal(cache_bits(c.k_cache), kc) and np.array_equal(cache_bits(c.v_cache), vc)
    ref = oracle.attention(case.q, kc, vc, case.block_table, case.context_lens, None, case.scale,
                           64, 8, case.num_pages, case.max_pages_per_seq)
    assert_close(out, ref, what="32b ragged")


EDGE = [1, 63, 64, 65, 127, 128, 129, 2051, 4096]


@pytest.mark.parametrize("Hq,Hkv", [(8, 1), (40, 8), (16, 16), (64, 8), (96, 8), (12, 2), (32, 2), (16, 1)])
def test_edge_lengths_and_groups(cuda_lib, Hq, Hkv):
    case = W.custom_case(400 + Hq, EDGE, Hq=Hq, Hkv=Hkv, max_pages_per_seq=32)
    for splits in (0, 1, 5):
        out, st = _decode(cuda_lib, case.to("cuda"), splits)
        assert st == 0
        assert_close(out, oracle_decode(case), what=f"edge Hq={Hq} Hkv={Hkv} s={splits}")


def test_zero_context_rows_are_exactly_zero(cuda_lib):
    case = W.custom_case(410, [0, 300, 0, 1], Hq=8, Hkv=2)
    for splits in (1, 2, BAL):
        out, st = _decode(cuda_lib, case.to("cuda"), splits)
        assert st == 0
        assert torch.count_nonzero(out[0]) == 0 and torch.count_nonzero(out[2]) == 0
        assert_close(out, oracle_decode(case), what="zero ctx")


@pytest.mark.parametrize("splits", [3, BAL])
def test_page_permutation_gives_bitwise_identical_output(cuda_lib, splits):
    case = W.custom_case(411, [300, 129, 4000, 17], Hq=40, Hkv=8, extra_pages=9,
                         max_pages_per_seq=32)
    base, _ = _decode(cuda_lib, case.to("cuda"), splits)
    perm = torch.randperm(case.num_pages, generator=torch.Generator().manual_seed(5))
    inv = torch.empty_like(perm); inv[perm] = torch.arange(case.num_pages)
    case.k_cache, case.v_cache = case.k_cache[perm], case.v_cache[perm]
    m = case.block_table >= 0
    case.block_table[m] = inv[case.block_table[m].long()].to(torch.int32)
    again, _ = _decode(cuda_lib, case.to("cuda"), splits)
    assert torch.equal(base, again)


def test_shared_prefix_pages(cuda_lib):
    case = W.custom_case(412, [700, 700], Hq=8, Hkv=2)
    case.block_table[1] = case.block_table[0]
    case.q[1] = case.q[0]
    out, st = _decode(cuda_lib, case.to("cuda"))
    assert st == 0 and torch.equal(out[0], out[1])


@pytest.mark.parametrize("splits", [1, 2, BAL])
def test_invalid_page_zeroes_sequence_and_flags(cuda_lib, splits):
    case = W.custom_case(413, [300, 300], Hq=8, Hkv=2)
    ref = oracle_decode(case)
    case.block_table[0, 2] = -1
    out, st = _decode(cuda_lib, case.to("cuda"), splits)
    assert st & cuda_lib.PA_STATUS_BAD_PAGE
    assert torch.count_nonzero(out[0]) == 0
    assert_close(out[1], ref[1], what="valid neighbour")


@pytest.mark.parametrize("splits", [1, BAL])
def test_context_too_long_flags_length(cuda_lib, splits):
    case = W.custom_case(414, [10, 200], Hq=4, Hkv=1)
    ref = oracle_decode(case)
    case.context_lens[0] = case.max_pages_per_seq * 128 + 1
    out, st = _decode(cuda_lib, case.to("cuda"), splits)
    assert st & cuda_lib.PA_STATUS_BAD_LENGTH
    assert torch.count_nonzero(out[0]) == 0
    assert_close(out[1], ref[1], what="valid neighbour")


def test_repeated_calls_are_deterministic(cuda_lib):
    case = W.qwen3_14b_decode_b16().to("cuda")
    a, _ = _decode(cuda_lib, case, 0)
    b, _ = _decode(cuda_lib, case, 0)
    assert torch.equal(a, b)


# ---- page-balanced schedule: cut units, empty ranges, empty sequences

def test_balanced_one_unit_cut_into_one_page_pieces(cuda_lib):
    """One (sequence, KV head) of 32 pages: the launch has 32 CTAs of one page
    each, so the combine merges 32 partial records."""
    case = W.custom_case(420, [4096], Hq=8, Hkv=1, max_pages_per_seq=32)
    out, st = _decode(cuda_lib, case.to("cuda"), BAL)
    assert st == 0
    assert_close(out, oracle_decode(case), what="one unit, 32 pieces")


def test_balanced_more_ctas_than_pages(cuda_lib):
    """Fewer pages than CTAs: many CTAs have an empty range."""
    case = W.custom_case(421, [8000, 3, 0], Hq=4, Hkv=1, max_pages_per_seq=63)
    out, st = _decode(cuda_lib, case.to("cuda"), BAL)
    assert st == 0
    assert torch.count_nonzero(out[2]) == 0
    assert_close(out, oracle_decode(case), what="empty CTA ranges")


def test_balanced_empty_sequences_everywhere(cuda_lib):
    """Empty contexts first, between and last (the last CTA owns position W)."""
    ctx = [0, 5, 0, 0, 1300, 129, 0, 2051, 0]
    case = W.custom_case(422, ctx, Hq=16, Hkv=2, max_pages_per_seq=17)
    out, st = _decode(cuda_lib, case.to("cuda"), BAL)
    assert st == 0
    for s, c in enumerate(ctx):
        if c == 0:
            assert torch.count_nonzero(out[s]) == 0
    assert_close(out, oracle_decode(case), what="empty sequences")


def test_balanced_largest_batch(cuda_lib):
    lens = torch.randint(1, 400, (cuda_lib.PA_BALANCED_MAX_SEQS,),
                         generator=torch.Generator().manual_seed(423)).tolist()
    lens[7] = 0
    case = W.custom_case(423, lens, Hq=4, Hkv=2, max_pages_per_seq=4)
    out, st = _decode(cuda_lib, case.to("cuda"), BAL)
    assert st == 0
    assert_close(out, oracle_decode(case), what="largest balanced batch")


def test_balanced_rejects_too_many_sequences(cuda_lib):
    case = W.custom_case(424, [3] * (cuda_lib.PA_BALANCED_MAX_SEQS + 1), Hq=2, Hkv=1,
                         max_pages_per_seq=1).to("cuda")
    d = cuda_lib.make_dims(case.B, case.Hq, case.Hkv, case.num_pages, case.max_pages_per_seq)
    assert cuda_lib.load().pa_decode_workspace_size(d, BAL) == 2**64 - 1
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    out = torch.empty(case.B, case.Hq, 128, dtype=torch.float32, device="cuda")
    rc = cuda_lib.load().pa_decode(
        cuda_lib._ptr(case.q), cuda_lib._ptr(case.k_cache), cuda_lib._ptr(case.v_cache),
        cuda_lib._ptr(case.block_table), cuda_lib._ptr(case.context_lens), case.scale,
        cuda_lib._ptr(out), cuda_lib.PA_F32, cuda_lib._ptr(ws), ws.numel(), BAL, d, None, None)
    assert rc == cuda_lib.PA_ERR_SPLITS
    # the automatic choice falls back to fixed splits for that batch
    out, st = _decode(cuda_lib, case, 0)
    assert st == 0
