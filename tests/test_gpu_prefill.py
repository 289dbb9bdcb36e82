"""pa_kv_write + pa_prefill_chunk on the GPU against the FP64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from pa_testutil import (assert_close, assert_close_bf16, cache_bits, dev_status,
                         oracle_prefill, sample_rows)

pytestmark = pytest.mark.gpu


def _write_and_prefill(pa, case, out_dtype=torch.float32):
    c = case.to("cuda")
    st = dev_status()
    pa.pa_kv_write(c.k_new, c.v_new, c.k_cache, c.v_cache, c.block_table, c.context_lens,
                   c.chunk_lens, status=st)
    out = pa.pa_prefill_chunk(c.q, c.k_cache, c.v_cache, c.block_table, c.context_lens,
                              c.chunk_lens, c.scale, out_dtype=out_dtype, status=st)
    torch.cuda.synchronize()
    return c, out, int(st.item())


def _oracle_after_write(case, rows=None):
    kc, vc, sk = oracle.kv_write(case.k_new, case.v_new, case.k_cache, case.v_cache,
                                 case.block_table, case.context_lens, case.chunk_lens,
                                 case.num_pages, case.max_pages_per_seq)
    ref = oracle.attention(case.q, kc, vc, case.block_table, case.context_lens, case.chunk_lens,
                           case.scale, case.Hq, case.Hkv, case.num_pages, case.max_pages_per_seq,
                           rows=rows)
    return ref, kc, vc


@pytest.mark.parametrize("ctx,chunk", [
    ([130, 5, 300], [3, 5, 129]),
    ([1, 257, 128, 129], [1, 257, 128, 1]),
    ([600, 300], [512, 300]),             # no prior context for the second sequence
    ([255, 1000], [127, 129]),
])
def test_small_cases_all_rows(cuda_lib, ctx, chunk):
    case = W.custom_case(500 + sum(chunk), ctx, Hq=8, Hkv=2, chunk_lens=chunk, with_new=True)
    c, out, st = _write_and_prefill(cuda_lib, case)
    assert st == 0
    ref, kc, _ = _oracle_after_write(case)
    assert np.array_equal(cache_bits(c.k_cache), kc)
    assert_close(out, ref, what=f"prefill ctx={ctx} chunk={chunk}")


@pytest.mark.parametrize("Hq,Hkv", [(40, 8), (64, 8), (8, 8), (16, 1), (12, 4)])
def test_head_layouts(cuda_lib, Hq, Hkv):
    case = W.custom_case(520 + Hq, [700, 129], Hq=Hq, Hkv=Hkv, chunk_lens=[200, 129],
                         with_new=True)
    _, out, st = _write_and_prefill(cuda_lib, case)
    assert st == 0
    ref, _, _ = _oracle_after_write(case)
    assert_close(out, ref, what=f"prefill Hq={Hq} Hkv={Hkv}")


def test_bf16_output(cuda_lib):
    case = W.custom_case(530, [900, 400], Hq=8, Hkv=2, chunk_lens=[300, 400], with_new=True)
    _, out, st = _write_and_prefill(cuda_lib, case, torch.bfloat16)
    assert st == 0
    ref, _, _ = _oracle_after_write(case)
    assert_close_bf16(out, ref, what="prefill bf16")


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_chunked_prefill_workload_sampled(cuda_lib, out_dtype):
    """The 8 x 512 chunked-prefill workload at full size (the benchmark's launch
    configuration, BF16 out: full 128-row tiles leave through TMA stores),
    checked on sampled (token, head) rows."""
    case = W.chunked_prefill()
    _, out, st = _write_and_prefill(cuda_lib, case, out_dtype)
    assert st == 0
    extra = []
    for s in range(8):   # first and last token of every sequence, a few heads
        for tok in (s * 512, s * 512 + 511, s * 512 + 127, s * 512 + 128):
            extra += [tok * 40 + h for h in (0, 4, 5, 39)]
    rows = sample_rows(case.T, 40, 600, seed=3, extra=extra)
    ref, _, _ = _oracle_after_write(case, rows=rows)
    got = out.reshape(-1, 128)[torch.as_tensor(rows, device="cuda")]
    if out_dtype == torch.float32:
        assert_close(got, ref, what="chunked prefill sampled")
    else:
        assert_close_bf16(got, ref, what="chunked prefill sampled, bf16 out")


def test_single_token_prefill_equals_decode(cuda_lib):
    case = W.custom_case(540, [300, 129, 1], Hq=40, Hkv=8, chunk_lens=[1, 1, 1], with_new=True)
    c, out, st = _write_and_prefill(cuda_lib, case)
    dec = cuda_lib.pa_decode(c.q, c.k_cache, c.v_cache, c.block_table, c.context_lens, c.scale,
                             out_dtype=torch.float32, num_splits=1)
    torch.cuda.synchronize()
    assert st == 0
    assert (out - dec).abs().max().item() < 2e-3


def test_last_prefill_row_equals_decode(cuda_lib):
    case = W.custom_case(541, [700, 300], Hq=8, Hkv=2, chunk_lens=[150, 44], with_new=True)
    c, out, st = _write_and_prefill(cuda_lib, case)
    q_last = torch.stack([c.q[149], c.q[193]])
    dec = cuda_lib.pa_decode(q_last, c.k_cache, c.v_cache, c.block_table, c.context_lens,
                             c.scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert st == 0
    assert (out[[149, 193]] - dec).abs().max().item() < 2e-3


def test_invalid_page_zeroes_sequence(cuda_lib):
    case = W.custom_case(542, [400, 400], Hq=8, Hkv=2, chunk_lens=[100, 100], with_new=True)
    ref, _, _ = _oracle_after_write(case)
    c = case.to("cuda")
    st = dev_status()
    cuda_lib.pa_kv_write(c.k_new, c.v_new, c.k_cache, c.v_cache, c.block_table, c.context_lens,
                         c.chunk_lens, status=st)
    c.block_table[0, 1] = 10 ** 6
    out = cuda_lib.pa_prefill_chunk(c.q, c.k_cache, c.v_cache, c.block_table, c.context_lens,
                                    c.chunk_lens, c.scale, out_dtype=torch.float32, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & cuda_lib.PA_STATUS_BAD_PAGE
    assert torch.count_nonzero(out[:100]) == 0
    assert_close(out[100:], ref[100:], what="valid neighbour")


def test_token_count_mismatch_flags(cuda_lib):
    case = W.custom_case(543, [300, 300], Hq=8, Hkv=2, chunk_lens=[100, 100], with_new=True)
    c = case.to("cuda")
    st = dev_status()
    cuda_lib.pa_prefill_chunk(c.q[:150], c.k_cache, c.v_cache, c.block_table, c.context_lens,
                              c.chunk_lens, c.scale, out_dtype=torch.float32, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & cuda_lib.PA_STATUS_BAD_TOKENS


def test_page_permutation_bitwise(cuda_lib):
    case = W.custom_case(544, [1000, 333], Hq=8, Hkv=2, chunk_lens=[260, 77], with_new=True,
                         extra_pages=5)
    _, base, _ = _write_and_prefill(cuda_lib, case)
    perm = torch.randperm(case.num_pages, generator=torch.Generator().manual_seed(9))
    inv = torch.empty_like(perm); inv[perm] = torch.arange(case.num_pages)
    case.k_cache, case.v_cache = case.k_cache[perm], case.v_cache[perm]
    m = case.block_table >= 0
    case.block_table[m] = inv[case.block_table[m].long()].to(torch.int32)
    _, again, _ = _write_and_prefill(cuda_lib, case)
    assert torch.equal(base, again)


@pytest.mark.parametrize("profile", ["ramp", "jump", "fall"])
def test_scores_that_move_the_reference(cuda_lib, profile):
    """Online softmax with a lazily moved reference: scores that rise by about
    ten octaves per 32-key chunk (every chunk moves the running reference, so
    P already in tensor memory, the partial sum, O and l are rescaled), one
    jump of about 130 octaves in the middle of a chunk (the old state scales
    to zero), and falling scores (the first chunk's maximum stays the
    reference).  The normalised output does not depend on the reference."""
    n = 700
    case = W.custom_case(611, [n], Hq=8, Hkv=2, chunk_lens=[n], with_new=True)
    j = torch.arange(n, dtype=torch.float32)
    f = {"ramp": 0.02 * j,
         "jump": torch.where(j >= 317, torch.full_like(j, 8.0), torch.zeros_like(j)),
         "fall": -0.02 * j}[profile]
    # q = 1 and k_j = f(j) in every dimension: c * q.k_j = 128 f(j) / sqrt(128) * log2(e)
    case.q = torch.ones_like(case.q)
    case.k_new = (f[:, None, None] * torch.ones(1, case.Hkv, 128)).to(torch.bfloat16)
    _, out, st = _write_and_prefill(cuda_lib, case)
    assert st == 0
    ref, _, _ = _oracle_after_write(case)
    assert_close(out, ref, what=f"prefill {profile} scores")


@pytest.mark.parametrize("extra", [-1, 2])
def test_schedule_table_limit(cuda_lib, extra):
    """Launches whose item count sits just below or just above what the
    per-pair schedule table holds (PA_PREFILL_SCHEDULE_ITEMS items per CTA
    pair, pa_prefill_pairs() pairs): below it every pair takes its items from
    the table, above it every pair falls back to round-robin -- never a mix,
    which would leave items unprocessed.  One pair of query tiles per sequence
    and 8 query heads, so items = 8 * sequences; the output starts as NaN and
    every row must be written."""
    pairs = cuda_lib.pa_prefill_pairs()
    B = cuda_lib.PA_PREFILL_SCHEDULE_ITEMS * pairs // 8 + extra
    chunk = [1 + s % 3 for s in range(B)]
    ctx = [c + (37 * s) % 150 for s, c in enumerate(chunk)]
    case = W.custom_case(612, ctx, Hq=8, Hkv=2, chunk_lens=chunk, with_new=True)
    c = case.to("cuda")
    st = dev_status()
    cuda_lib.pa_kv_write(c.k_new, c.v_new, c.k_cache, c.v_cache, c.block_table, c.context_lens,
                         c.chunk_lens, status=st)
    out = torch.full((sum(chunk), 8, 128), float("nan"), dtype=torch.float32, device="cuda")
    cuda_lib.pa_prefill_chunk(c.q, c.k_cache, c.v_cache, c.block_table, c.context_lens,
                              c.chunk_lens, c.scale, out=out, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert bool(torch.isfinite(out).all()), "rows left unwritten"
    T = sum(chunk)
    rows = sample_rows(T, 8, 200, seed=13, extra=[0, 8 * T - 1, 8 * (T // 2) + 3])
    ref, _, _ = _oracle_after_write(case, rows=rows)
    got = out.reshape(-1, 128)[torch.as_tensor(rows, device="cuda")]
    assert_close(got, ref, what=f"schedule limit B={B}")
