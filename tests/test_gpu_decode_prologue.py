"""pa_decode_prologue (the decode step with its QK-norm / RoPE / KV-write
prologue inside the attention kernel) on the GPU.

Its result is defined as that of pa_qk_norm_rope_write followed by pa_decode:
checked bit for bit against that pair (output, both caches, status bits) on
head layouts, schedules, invalid and empty sequences and the full batch-128 x
4096 step; and the chain against the FP64 oracle (oracle prologue, then
oracle attention)."""
import math

import pytest
import torch

import oracle
import workloads as W
from pa_testutil import assert_close, dev_status

pytestmark = pytest.mark.gpu
D = 128


def _two_calls(pa, c, qkv, wq, wk, splits, out_dtype=torch.float32, **kw):
    kc, vc = c.k_cache.clone(), c.v_cache.clone()
    st = dev_status()
    q = pa.pa_qk_norm_rope_write(qkv, wq, wk, kc, vc, c.block_table, c.context_lens, None,
                                 status=st, **kw)
    out = pa.pa_decode(q, kc, vc, c.block_table, c.context_lens, 1.0, out_dtype=out_dtype,
                       num_splits=splits, status=st)
    torch.cuda.synchronize()
    return out, kc, vc, int(st.item())


def _fused(pa, c, qkv, wq, wk, splits, out_dtype=torch.float32, **kw):
    kc, vc = c.k_cache.clone(), c.v_cache.clone()
    st = dev_status()
    out = pa.pa_decode_prologue(qkv, wq, wk, kc, vc, c.block_table, c.context_lens, scale=1.0,
                                out_dtype=out_dtype, num_splits=splits, status=st, **kw)
    torch.cuda.synchronize()
    return out, kc, vc, int(st.item())


def _same(a, b, what):
    out_a, kc_a, vc_a, st_a = a
    out_b, kc_b, vc_b, st_b = b
    assert st_a == st_b, f"{what}: status {st_a} != {st_b}"
    assert torch.equal(out_a.view(torch.int32) if out_a.dtype == torch.float32 else out_a.view(torch.int16),
                       out_b.view(torch.int32) if out_b.dtype == torch.float32 else out_b.view(torch.int16)), \
        f"{what}: outputs differ (max {(out_a.float() - out_b.float()).abs().max().item():.3e})"
    assert torch.equal(kc_a.view(torch.int16), kc_b.view(torch.int16)), f"{what}: K caches differ"
    assert torch.equal(vc_a.view(torch.int16), vc_b.view(torch.int16)), f"{what}: V caches differ"


def _inputs(c, seed):
    qkv, wq, wk = W.prologue_inputs(c, seed)
    return qkv.cuda(), wq.cuda(), wk.cuda()


@pytest.mark.parametrize("hq,hkv", [(40, 8), (64, 8), (8, 1), (16, 16), (32, 2)])
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_fused_equals_prologue_then_decode(cuda_lib, hq, hkv, splits):
    ctx = [1, 200, 4096, 37, 129, 128]
    c = W.custom_case(700 + hq + hkv, ctx, Hq=hq, Hkv=hkv, max_pages_per_seq=32).to("cuda")
    qkv, wq, wk = _inputs(c, 700 + hq)
    kw = dict(eps=1e-6, rope_base=1e6, rope_scale=1.0, q_scale=1.0 / math.sqrt(D))
    a = _two_calls(cuda_lib, c, qkv, wq, wk, splits, **kw)
    b = _fused(cuda_lib, c, qkv, wq, wk, splits, **kw)
    assert a[3] == 0
    _same(a, b, f"{hq}/{hkv} splits={splits}")


def test_bf16_out_long_positions_and_rope_scaling(cuda_lib):
    """Positions up to 32767 (the double-precision angle path past 2^22 turns
    of the fastest pair) with a non-unit frequency divisor, BF16 output."""
    c = W.custom_case(710, [32768, 20000, 1], Hq=8, Hkv=2, max_pages_per_seq=256,
                      extra_pages=2).to("cuda")
    qkv, wq, wk = _inputs(c, 710)
    for base, scale in ((1e6, 1.0), (1e4, 4.0)):
        kw = dict(eps=1e-5, rope_base=base, rope_scale=scale)
        a = _two_calls(cuda_lib, c, qkv, wq, wk, 0, out_dtype=torch.bfloat16, **kw)
        b = _fused(cuda_lib, c, qkv, wq, wk, 0, out_dtype=torch.bfloat16, **kw)
        _same(a, b, f"base={base} scale={scale}")


@pytest.mark.parametrize("splits", [0, 1, 4])
def test_invalid_and_empty_sequences(cuda_lib, splits):
    """A block-table entry out of range early in a long sequence (the page
    holding its new token is valid and, under the page-balanced schedule, read
    by another CTA than the bad one), a length past the table and an empty
    sequence: same status bits, nothing written for them, zero rows."""
    ctx = [4096, 300, 0, 129, 4096]
    c = W.custom_case(720, ctx, Hq=40, Hkv=8, max_pages_per_seq=32)
    c.block_table[0, 3] = -7
    c.context_lens[3] = 32 * 128 + 1
    c = c.to("cuda")
    qkv, wq, wk = _inputs(c, 720)
    a = _two_calls(cuda_lib, c, qkv, wq, wk, splits)
    b = _fused(cuda_lib, c, qkv, wq, wk, splits)
    st = a[3]
    assert st & cuda_lib.PA_STATUS_BAD_PAGE and st & cuda_lib.PA_STATUS_BAD_LENGTH
    _same(a, b, f"invalid splits={splits}")
    for s in (0, 2, 3):
        assert torch.count_nonzero(b[0][s]) == 0


def test_full_size_b128_equals_two_calls(cuda_lib):
    """The benchmark's decode step shape: 128 sequences x 4096 tokens, 40/8 heads."""
    c = W.qwen3_14b_decode_b128(device="cuda", pool_device="cuda", with_new=False)
    qkv, wq, wk = W.prologue_inputs(c, 730, device="cuda")
    kw = dict(q_scale=1.0 / math.sqrt(D))
    a = _two_calls(cuda_lib, c, qkv, wq, wk, 0, out_dtype=torch.bfloat16, **kw)
    b = _fused(cuda_lib, c, qkv, wq, wk, 0, out_dtype=torch.bfloat16, **kw)
    assert a[3] == 0
    _same(a, b, "b128")


def test_fused_matches_the_oracle_chain(cuda_lib):
    """Against the oracle: its prologue (Q, and K/V written to the slots), then
    its attention over the written cache with Q rounded to bf16 (the GPU's
    operand), the softmax scale folded into Q."""
    ctx = [1, 513, 4096, 2051, 64, 128]
    c = W.custom_case(740, ctx, Hq=40, Hkv=8, max_pages_per_seq=32)
    qkv, wq, wk = W.prologue_inputs(c, 740)
    kw = dict(q_scale=1.0 / math.sqrt(D))
    cd = c.to("cuda")
    out, kc, vc, st = _fused(cuda_lib, cd, qkv.cuda(), wq.cuda(), wk.cuda(), 0, **kw)
    assert st == 0
    q_ref, k_ref, v_ref, skipped = oracle.qk_norm_rope_write(
        qkv, wq.numpy(), wk.numpy(), c.k_cache, c.v_cache, c.block_table, c.context_lens, None,
        c.Hq, c.Hkv, c.num_pages, c.max_pages_per_seq, **kw)
    assert skipped == 0
    qb = torch.from_numpy(q_ref).float().to(torch.bfloat16)
    ref = oracle.attention(qb, k_ref, v_ref, c.block_table, c.context_lens, None, 1.0,
                           c.Hq, c.Hkv, c.num_pages, c.max_pages_per_seq)
    assert_close(out, ref, what="fused prologue + decode")
