"""FP8 (e4m3) KV cache on the GPU: pa_kv_write_fp8 bit for bit against the
oracle's quantizing write, and pa_decode_fp8 against the oracle's FP64
attention over the dequantized cache."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from pa_testutil import assert_close, dev_status, sample_rows

pytestmark = pytest.mark.gpu

BAL = -1


def _scales(Hkv, seed):
    g = torch.Generator().manual_seed(seed)
    # N(0, 1) data / [0.02, 0.04]: codes stay inside +-448 (no saturation)
    ks = (torch.rand(Hkv, generator=g) * 0.02 + 0.02).float()
    vs = (torch.rand(Hkv, generator=g) * 0.02 + 0.02).float()
    return ks, vs


def _quantize_cache(cache, scale):
    """Starting FP8 cache (an input): every cached bf16 value / scale[h] as e4m3
    through torch's float8_e4m3fn conversion, which the oracle pins equal to its
    own encoder inside +-448; NaN-poisoned slots stay NaN codes."""
    x = cache.float() / scale[None, None, :, None]
    return x.to(torch.float8_e4m3fn).view(torch.uint8)


def _fp8_case(case, seed):
    ks, vs = _scales(case.Hkv, seed)
    return ks, vs, _quantize_cache(case.k_cache, ks), _quantize_cache(case.v_cache, vs)


def _run(pa, case, ks, vs, kc8, vc8, q_len=1, splits=0, out_dtype=torch.float32):
    c = case.to("cuda")
    kc, vc = kc8.cuda(), vc8.cuda()
    ksd, vsd = ks.cuda(), vs.cuda()
    st = dev_status()
    if case.k_new is not None:
        pa.pa_kv_write_fp8(c.k_new, c.v_new, kc, vc, ksd, vsd, c.block_table, c.context_lens,
                           c.chunk_lens, status=st)
    out = pa.pa_decode_fp8(c.q, kc, vc, ksd, vsd, c.block_table, c.context_lens, q_len,
                           c.scale, out_dtype=out_dtype, num_splits=splits, status=st)
    torch.cuda.synchronize()
    return out, kc.cpu().numpy(), vc.cpu().numpy(), int(st.item())


def _oracle(case, ks, vs, kc8, vc8, rows=None):
    kc, vc = kc8.numpy(), vc8.numpy()
    if case.k_new is not None:
        kc, vc, _ = oracle.kv_write_fp8(case.k_new, case.v_new, kc, vc, ks, vs, case.block_table,
                                        case.context_lens, case.chunk_lens, case.num_pages,
                                        case.max_pages_per_seq)
    ref = oracle.attention_fp8(case.q, kc, vc, ks, vs, case.block_table, case.context_lens,
                               case.chunk_lens, case.scale, case.Hq, case.Hkv, case.num_pages,
                               case.max_pages_per_seq, rows=rows)
    return ref, kc, vc


@pytest.mark.parametrize("chunk", [None, [3, 129, 1, 200]])
def test_kv_write_fp8_bitwise(cuda_lib, chunk):
    ctx = [300, 129, 1, 700]
    case = W.custom_case(801, ctx, Hq=8, Hkv=2, chunk_lens=chunk, with_new=True)
    ks, vs, kc8, vc8 = _fp8_case(case, 1)
    c = case.to("cuda")
    kc, vc = kc8.cuda(), vc8.cuda()
    st = dev_status()
    cuda_lib.pa_kv_write_fp8(c.k_new, c.v_new, kc, vc, ks.cuda(), vs.cuda(), c.block_table,
                             c.context_lens, c.chunk_lens, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    _, rk, rv = _oracle(case, ks, vs, kc8, vc8, rows=np.array([0]))
    assert np.array_equal(kc.cpu().numpy(), rk)
    assert np.array_equal(vc.cpu().numpy(), rv)


@pytest.mark.parametrize("splits", [0, 1, 3, BAL])
def test_decode_fp8_ragged(cuda_lib, splits):
    ctx = [1, 130, 4096, 777, 129, 2000]
    case = W.custom_case(810, ctx, Hq=40, Hkv=8, with_new=True)
    ks, vs, kc8, vc8 = _fp8_case(case, 2)
    out, kc, vc, st = _run(cuda_lib, case, ks, vs, kc8, vc8, splits=splits)
    assert st == 0
    ref, rk, rv = _oracle(case, ks, vs, kc8, vc8)
    assert np.array_equal(kc, rk) and np.array_equal(vc, rv)
    assert_close(out, ref, what=f"fp8 decode splits={splits}")


@pytest.mark.parametrize("Hq,Hkv,q_len", [(8, 2, 1), (64, 8, 1), (16, 1, 1), (40, 8, 2),
                                          (40, 8, 4), (64, 8, 3)])
def test_decode_fp8_layouts_and_q_len(cuda_lib, Hq, Hkv, q_len):
    ctx = [700, 129, q_len, 1500]
    case = W.custom_case(820 + Hq + q_len, ctx, Hq=Hq, Hkv=Hkv, chunk_lens=[q_len] * 4,
                         with_new=True)
    ks, vs, kc8, vc8 = _fp8_case(case, 3)
    out, _, _, st = _run(cuda_lib, case, ks, vs, kc8, vc8, q_len=q_len)
    assert st == 0
    ref, _, _ = _oracle(case, ks, vs, kc8, vc8)
    assert_close(out, ref, what=f"fp8 Hq={Hq} Hkv={Hkv} q_len={q_len}")


def test_decode_fp8_bf16_output(cuda_lib):
    case = W.custom_case(830, [900, 33], Hq=40, Hkv=8, with_new=True)
    ks, vs, kc8, vc8 = _fp8_case(case, 4)
    out, _, _, st = _run(cuda_lib, case, ks, vs, kc8, vc8, out_dtype=torch.bfloat16)
    assert st == 0
    ref, _, _ = _oracle(case, ks, vs, kc8, vc8)
    g = out.float().cpu().double().numpy()
    assert (np.abs(g - ref) <= 5e-3 + np.abs(ref) * 2.0 ** -8).all()


def test_decode_fp8_q_beyond_f16_range(cuda_lib):
    """q . K runs on e4m3 codes with q split into hi + lo after scaling by a
    power of two per work item, so no bf16 magnitude is out of range: q times
    2^15 (elements past 65520) with the softmax scale times 2^-15 gives the
    same codes, the same score factor and so the same bits as the unscaled
    call, which matches the oracle."""
    case = W.custom_case(840, [300, 200, 4096], Hq=8, Hkv=2, with_new=True)
    ks, vs, kc8, vc8 = _fp8_case(case, 5)
    out, _, _, st = _run(cuda_lib, case, ks, vs, kc8, vc8)
    assert st == 0
    ref, _, _ = _oracle(case, ks, vs, kc8, vc8)
    assert_close(out, ref, what="fp8 unscaled q")
    big = W.custom_case(840, [300, 200, 4096], Hq=8, Hkv=2, with_new=True)
    big.q = (big.q.float() * 2.0 ** 15).to(torch.bfloat16)
    big.scale = case.scale * 2.0 ** -15
    assert big.q.float().abs().max() > 65520
    out_big, _, _, st = _run(cuda_lib, big, ks, vs, kc8, vc8)
    assert st == 0
    assert torch.equal(out_big.view(torch.int32), out.view(torch.int32))


def test_decode_fp8_q_wide_dynamic_range(cuda_lib):
    """Elements far below their row's largest (down to 2^-16 of it), where the
    hi + lo split is no longer exact (error at most 2^-17 of the largest):
    still within the tolerance of the oracle."""
    case = W.custom_case(845, [777, 4096, 129], Hq=40, Hkv=8, with_new=True)
    g = torch.Generator().manual_seed(845)
    e = torch.randint(-16, 1, case.q.shape, generator=g).float()
    case.q = (case.q.float() * torch.exp2(e) * 4.0).to(torch.bfloat16)
    ks, vs, kc8, vc8 = _fp8_case(case, 7)
    out, _, _, st = _run(cuda_lib, case, ks, vs, kc8, vc8)
    assert st == 0
    ref, _, _ = _oracle(case, ks, vs, kc8, vc8)
    assert_close(out, ref, what="fp8 wide-range q")


def test_decode_fp8_nonfinite_q_is_flagged(cuda_lib):
    """An infinite q element sets PA_STATUS_Q_RANGE and its work item's rows
    come out NaN; the other sequence is unaffected."""
    case = W.custom_case(846, [300, 200], Hq=8, Hkv=2, with_new=True)
    ks, vs, kc8, vc8 = _fp8_case(case, 5)
    case.q[1, 3, 17] = float("inf")
    out, _, _, st = _run(cuda_lib, case, ks, vs, kc8, vc8, splits=1)
    assert st & cuda_lib.PA_STATUS_Q_RANGE
    assert torch.isnan(out[1, 0:4]).all()  # query heads 0-3 share KV head 0
    ref, _, _ = _oracle(case, ks, vs, kc8, vc8)
    assert_close(out[0:1], ref[0:1], what="fp8 other sequence")


def test_decode_fp8_full_size_sampled(cuda_lib):
    """The benchmark's FP8 workload: 128 sequences x 4096 tokens, 40/8 heads,
    e4m3 K/V (1.07 GB), the automatic schedule; sampled rows."""
    case = W.qwen3_14b_decode_b128(with_new=True)
    ks, vs, kc8, vc8 = _fp8_case(case, 6)
    out, _, _, st = _run(cuda_lib, case, ks, vs, kc8, vc8)
    assert st == 0
    rows = sample_rows(128, 40, 64, seed=5, extra=[41, 5000])
    ref, _, _ = _oracle(case, ks, vs, kc8, vc8, rows=rows)
    got = out.reshape(-1, 128)[torch.as_tensor(rows, device="cuda")]
    assert_close(got, ref, what="fp8 b128 sampled")
