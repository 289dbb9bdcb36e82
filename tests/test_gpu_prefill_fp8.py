"""Chunked prefill over an FP8 (e4m3) cache on the GPU: pa_kv_write_fp8 +
pa_prefill_chunk_fp8 against the oracle's quantizing write and its FP64
causal attention over the dequantized cache (codes times the per-KV-head
scales), at the same tolerance as every other attention test."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from pa_testutil import assert_close, assert_close_bf16, dev_status, sample_rows

pytestmark = pytest.mark.gpu


def _scales(Hkv, seed):
    g = torch.Generator().manual_seed(seed)
    # N(0, 1) data / [0.02, 0.04]: codes stay inside +-448 (no saturation)
    ks = (torch.rand(Hkv, generator=g) * 0.02 + 0.02).float()
    vs = (torch.rand(Hkv, generator=g) * 0.02 + 0.02).float()
    return ks, vs


def _quantize_cache(cache, scale):
    """Starting FP8 cache (an input): every cached bf16 value / scale[h] as e4m3
    through torch's float8_e4m3fn conversion (the oracle's encoder is pinned to
    it inside +-448); NaN-poisoned slots stay NaN codes."""
    x = cache.float() / scale[None, None, :, None]
    return x.to(torch.float8_e4m3fn).view(torch.uint8)


def _fp8_case(case, seed):
    ks, vs = _scales(case.Hkv, seed)
    return ks, vs, _quantize_cache(case.k_cache, ks), _quantize_cache(case.v_cache, vs)


def _write_and_prefill(pa, case, ks, vs, kc8, vc8, out_dtype=torch.float32, q=None):
    c = case.to("cuda")
    kc, vc = kc8.cuda(), vc8.cuda()
    ksd, vsd = ks.cuda(), vs.cuda()
    st = dev_status()
    pa.pa_kv_write_fp8(c.k_new, c.v_new, kc, vc, ksd, vsd, c.block_table, c.context_lens,
                       c.chunk_lens, status=st)
    out = pa.pa_prefill_chunk_fp8(c.q if q is None else q, kc, vc, ksd, vsd, c.block_table,
                                  c.context_lens, c.chunk_lens, c.scale, out_dtype=out_dtype,
                                  status=st)
    torch.cuda.synchronize()
    return out, kc.cpu().numpy(), int(st.item())


def _oracle(case, ks, vs, kc8, vc8, rows=None):
    kc, vc, _ = oracle.kv_write_fp8(case.k_new, case.v_new, kc8.numpy(), vc8.numpy(), ks, vs,
                                    case.block_table, case.context_lens, case.chunk_lens,
                                    case.num_pages, case.max_pages_per_seq)
    ref = oracle.attention_fp8(case.q, kc, vc, ks, vs, case.block_table, case.context_lens,
                               case.chunk_lens, case.scale, case.Hq, case.Hkv, case.num_pages,
                               case.max_pages_per_seq, rows=rows)
    return ref, kc


@pytest.mark.parametrize("ctx,chunk", [
    ([130, 5, 300], [3, 5, 129]),
    ([1, 257, 128, 129], [1, 257, 128, 1]),
    ([600, 300], [512, 300]),             # no prior context for the second sequence
    ([255, 1000], [127, 129]),
])
def test_small_cases_all_rows(cuda_lib, ctx, chunk):
    case = W.custom_case(900 + sum(chunk), ctx, Hq=8, Hkv=2, chunk_lens=chunk, with_new=True)
    ks, vs, kc8, vc8 = _fp8_case(case, 11)
    out, kc, st = _write_and_prefill(cuda_lib, case, ks, vs, kc8, vc8)
    assert st == 0
    ref, rk = _oracle(case, ks, vs, kc8, vc8)
    assert np.array_equal(kc, rk)
    assert_close(out, ref, what=f"prefill fp8 ctx={ctx} chunk={chunk}")


@pytest.mark.parametrize("Hq,Hkv", [(40, 8), (64, 8), (16, 1), (12, 4)])
def test_head_layouts(cuda_lib, Hq, Hkv):
    case = W.custom_case(920 + Hq, [700, 129], Hq=Hq, Hkv=Hkv, chunk_lens=[200, 129],
                         with_new=True)
    ks, vs, kc8, vc8 = _fp8_case(case, Hq)
    out, _, st = _write_and_prefill(cuda_lib, case, ks, vs, kc8, vc8)
    assert st == 0
    ref, _ = _oracle(case, ks, vs, kc8, vc8)
    assert_close(out, ref, what=f"prefill fp8 Hq={Hq} Hkv={Hkv}")


def test_bf16_output(cuda_lib):
    case = W.custom_case(930, [900, 400], Hq=8, Hkv=2, chunk_lens=[300, 400], with_new=True)
    ks, vs, kc8, vc8 = _fp8_case(case, 3)
    out, _, st = _write_and_prefill(cuda_lib, case, ks, vs, kc8, vc8, torch.bfloat16)
    assert st == 0
    ref, _ = _oracle(case, ks, vs, kc8, vc8)
    assert_close_bf16(out, ref, what="prefill fp8 bf16")


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_chunked_prefill_workload_sampled(cuda_lib, out_dtype):
    """The 8 x 512 chunked-prefill workload at full size over an FP8 cache (the
    benchmark's launch configuration), checked on sampled (token, head) rows."""
    case = W.chunked_prefill()
    ks, vs, kc8, vc8 = _fp8_case(case, 5)
    out, _, st = _write_and_prefill(cuda_lib, case, ks, vs, kc8, vc8, out_dtype)
    assert st == 0
    extra = []
    for s in range(8):   # first and last token of every sequence, a few heads
        for tok in (s * 512, s * 512 + 511, s * 512 + 127, s * 512 + 128):
            extra += [tok * 40 + h for h in (0, 4, 5, 39)]
    rows = sample_rows(case.T, 40, 500, seed=7, extra=extra)
    ref, _ = _oracle(case, ks, vs, kc8, vc8, rows=rows)
    got = out.reshape(-1, 128)[torch.as_tensor(rows, device="cuda")]
    if out_dtype == torch.float32:
        assert_close(got, ref, what="prefill fp8 sampled")
    else:
        assert_close_bf16(got, ref, what="prefill fp8 sampled, bf16 out")


def test_matches_decode_fp8_on_single_tokens(cuda_lib):
    """chunk_lens = 1: the same attention pa_decode_fp8 computes."""
    case = W.custom_case(940, [300, 129, 1], Hq=40, Hkv=8, chunk_lens=[1, 1, 1], with_new=True)
    ks, vs, kc8, vc8 = _fp8_case(case, 9)
    c = case.to("cuda")
    kc, vc = kc8.cuda(), vc8.cuda()
    ksd, vsd = ks.cuda(), vs.cuda()
    st = dev_status()
    cuda_lib.pa_kv_write_fp8(c.k_new, c.v_new, kc, vc, ksd, vsd, c.block_table, c.context_lens,
                             c.chunk_lens, status=st)
    pf = cuda_lib.pa_prefill_chunk_fp8(c.q, kc, vc, ksd, vsd, c.block_table, c.context_lens,
                                       c.chunk_lens, c.scale, out_dtype=torch.float32, status=st)
    dec = cuda_lib.pa_decode_fp8(c.q, kc, vc, ksd, vsd, c.block_table, c.context_lens, 1, c.scale,
                                 out_dtype=torch.float32, num_splits=1, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert (pf - dec).abs().max().item() < 2e-3


def test_invalid_page_zeroes_sequence(cuda_lib):
    case = W.custom_case(942, [400, 400], Hq=8, Hkv=2, chunk_lens=[100, 100], with_new=True)
    ks, vs, kc8, vc8 = _fp8_case(case, 13)
    ref, _ = _oracle(case, ks, vs, kc8, vc8)
    c = case.to("cuda")
    kc, vc = kc8.cuda(), vc8.cuda()
    ksd, vsd = ks.cuda(), vs.cuda()
    st = dev_status()
    cuda_lib.pa_kv_write_fp8(c.k_new, c.v_new, kc, vc, ksd, vsd, c.block_table, c.context_lens,
                             c.chunk_lens, status=st)
    c.block_table[0, 1] = 10 ** 6
    out = cuda_lib.pa_prefill_chunk_fp8(c.q, kc, vc, ksd, vsd, c.block_table, c.context_lens,
                                        c.chunk_lens, c.scale, out_dtype=torch.float32, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & cuda_lib.PA_STATUS_BAD_PAGE
    assert out[:100].abs().max().item() == 0.0
    assert_close(out[100:], ref[100:], what="prefill fp8 valid neighbour")


def test_q_beyond_f16_range(cuda_lib):
    """QK^T runs on the e4m3 K codes with each query row split into e4m3 hi +
    lo after scaling by a power of two of its own, so no bf16 magnitude is out
    of range: q times 2^15 (elements past 65520) with the softmax scale times
    2^-15 gives the same codes, the same score factor and so the same bits as
    the unscaled call, which matches the oracle."""
    case = W.custom_case(944, [300, 1000], Hq=8, Hkv=2, chunk_lens=[100, 260], with_new=True)
    ks, vs, kc8, vc8 = _fp8_case(case, 17)
    out, _, st = _write_and_prefill(cuda_lib, case, ks, vs, kc8, vc8)
    assert st == 0
    ref, _ = _oracle(case, ks, vs, kc8, vc8)
    assert_close(out, ref, what="prefill fp8 unscaled q")
    big = W.custom_case(944, [300, 1000], Hq=8, Hkv=2, chunk_lens=[100, 260], with_new=True)
    big.q = (big.q.float() * 2.0 ** 15).to(torch.bfloat16)
    big.scale = case.scale * 2.0 ** -15
    assert big.q.float().abs().max() > 65520
    out_big, _, st = _write_and_prefill(cuda_lib, big, ks, vs, kc8, vc8)
    assert st == 0
    assert torch.equal(out_big.view(torch.int32), out.view(torch.int32))


def test_q_wide_dynamic_range(cuda_lib):
    """Elements far below their row's largest (down to 2^-16 of it), where the
    hi + lo split is no longer exact (error at most 2^-17 of the largest):
    still within the tolerance of the oracle."""
    case = W.custom_case(945, [700, 129], Hq=40, Hkv=8, chunk_lens=[300, 129], with_new=True)
    g = torch.Generator().manual_seed(945)
    e = torch.randint(-16, 1, case.q.shape, generator=g).float()
    case.q = (case.q.float() * torch.exp2(e) * 4.0).to(torch.bfloat16)
    ks, vs, kc8, vc8 = _fp8_case(case, 18)
    out, _, st = _write_and_prefill(cuda_lib, case, ks, vs, kc8, vc8)
    assert st == 0
    ref, _ = _oracle(case, ks, vs, kc8, vc8)
    assert_close(out, ref, what="prefill fp8 wide-range q")


def test_nonfinite_q_sets_status(cuda_lib):
    """An infinite q element sets PA_STATUS_Q_RANGE (that row's output is NaN;
    the other sequence is still right)."""
    case = W.custom_case(946, [300, 300], Hq=8, Hkv=2, chunk_lens=[100, 100], with_new=True)
    ks, vs, kc8, vc8 = _fp8_case(case, 17)
    ref, _ = _oracle(case, ks, vs, kc8, vc8)
    q = case.q.clone().cuda()
    q[150, 3, 7] = float("inf")
    out, _, st = _write_and_prefill(cuda_lib, case, ks, vs, kc8, vc8, q=q)
    assert st & cuda_lib.PA_STATUS_Q_RANGE
    assert torch.isnan(out[150, 3]).all()
    assert_close(out[:100], ref[:100], what="prefill fp8 beside a non-finite q")
