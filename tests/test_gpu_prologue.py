"""pa_qk_norm_rope_write (per-head RMSNorm of Q and K, NeoX RoPE, KV cache
write) on the GPU against the FP64 oracle.  Q is compared within a BF16 rounding
of the oracle's exact value; K within one BF16 ulp of the oracle's rounded K
(the GPU computes in FP32); V and every untouched cache byte bit for bit."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from pa_testutil import assert_close, dev_status, oracle_decode

pytestmark = pytest.mark.gpu
D = 128


def _bf16_to_f64(t):
    return t.detach().float().cpu().double().numpy()


def _bits_to_f64(b):
    return (np.asarray(b, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def _check_q(q_gpu, q_ref, what):
    g = _bf16_to_f64(q_gpu)
    scale = np.abs(q_ref).max(axis=-1, keepdims=True) + 1e-30
    err = np.abs(g - q_ref)
    bad = err > 2.0 ** -8 * np.abs(q_ref) + 2.0 ** -11 * scale
    assert not bad.any(), f"{what}: {bad.sum()} q values off, max err {err.max():.3e}"


def _written_slots(c, chunked, skip=()):
    """(page, offset) of every new token of a valid sequence (the KV write's slots)."""
    out = []
    for s in range(c.B):
        if s in skip:
            continue
        ctx = int(c.context_lens[s])
        n = int(c.chunk_lens[s]) if chunked else 1
        for j in range(n):
            pos = ctx - n + j
            out.append((int(c.block_table[s, pos // 128]), pos % 128))
    return out


def _check_caches(c, k_gpu, v_gpu, k_ref_bits, v_ref_bits, what, chunked=False, skip=()):
    kg = k_gpu.detach().cpu().view(torch.int16).numpy().view(np.uint16)
    vg = v_gpu.detach().cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(vg, v_ref_bits), f"{what}: V cache differs"
    written = np.zeros(kg.shape[:2], dtype=bool)
    for page, off in _written_slots(c, chunked, skip):
        written[page, off] = True
    # every other row is untouched, bit for bit (NaN poison included)
    assert np.array_equal(kg[~written], oracle._u16(c.k_cache)[~written]), \
        f"{what}: K rows outside the new tokens' slots changed"
    assert np.array_equal(k_ref_bits[~written], oracle._u16(c.k_cache)[~written])
    a, b = _bits_to_f64(kg[written]), _bits_to_f64(k_ref_bits[written])  # [rows, Hkv, D]
    # one bf16 ulp, plus an absolute term for results near zero after the RoPE
    # rotation's cancellation (FP32 arithmetic on values of the head's magnitude)
    head = np.abs(b).max(axis=-1, keepdims=True)
    assert np.all(np.abs(a - b) <= 2.0 ** -7 * np.abs(b) + 2.0 ** -14 * head), \
        f"{what}: K rows differ by more than one bf16 ulp (max {np.abs(a - b).max():.3e})"


def _run(pa, c, qkv, wq, wk, chunk_lens=None, **kw):
    cd = c.to("cuda")
    st = dev_status()
    q = pa.pa_qk_norm_rope_write(qkv.cuda(), wq.cuda(), wk.cuda(), cd.k_cache, cd.v_cache,
                                 cd.block_table, cd.context_lens,
                                 None if chunk_lens is None else cd.chunk_lens, status=st, **kw)
    torch.cuda.synchronize()
    return q, cd, int(st.item())


def _oracle(c, qkv, wq, wk, chunk_lens=None, **kw):
    return oracle.qk_norm_rope_write(qkv, wq.numpy(), wk.numpy(), c.k_cache, c.v_cache,
                                     c.block_table, c.context_lens, chunk_lens, c.Hq, c.Hkv,
                                     c.num_pages, c.max_pages_per_seq, **kw)


@pytest.mark.parametrize("hq,hkv", [(40, 8), (64, 8), (8, 1), (16, 16)])
def test_decode_prologue(cuda_lib, hq, hkv):
    ctx = [1, 200, 4096, 37, 129, 128]
    c = W.custom_case(500 + hq, ctx, Hq=hq, Hkv=hkv, max_pages_per_seq=32)
    qkv, wq, wk = W.prologue_inputs(c, 500 + hq)
    kw = dict(eps=1e-6, rope_base=1e6, rope_scale=1.0, q_scale=1.0 / math.sqrt(D))
    q, cd, st = _run(cuda_lib, c, qkv, wq, wk, **kw)
    assert st == 0
    q_ref, k_ref, v_ref, skipped = _oracle(c, qkv, wq, wk, **kw)
    assert skipped == 0
    _check_q(q, q_ref, f"decode q {hq}/{hkv}")
    _check_caches(c, cd.k_cache, cd.v_cache, k_ref, v_ref, "decode")


def test_long_positions_and_rope_scaling(cuda_lib):
    """Positions up to 32767 (angles of thousands of radians) with a non-unit
    frequency divisor and base: the angle reduction must keep full accuracy."""
    ctx = [32768, 20000, 1]
    c = W.custom_case(510, ctx, Hq=8, Hkv=2, max_pages_per_seq=256, extra_pages=2)
    qkv, wq, wk = W.prologue_inputs(c, 510)
    for base, scale in ((1e6, 1.0), (1e4, 4.0), (5e5, 0.5)):
        kw = dict(eps=1e-5, rope_base=base, rope_scale=scale)
        q, cd, st = _run(cuda_lib, c, qkv, wq, wk, **kw)
        assert st == 0
        q_ref, k_ref, v_ref, _ = _oracle(c, qkv, wq, wk, **kw)
        _check_q(q, q_ref, f"long positions base={base} scale={scale}")
        _check_caches(c, cd.k_cache, cd.v_cache, k_ref, v_ref, "long")


def test_chunked_prefill_prologue_full_size(cuda_lib):
    """The benchmark's chunked prefill: 8 sequences x 512 new tokens (T = 4096)."""
    c = W.chunked_prefill()
    qkv, wq, wk = W.prologue_inputs(c, 520)
    q, cd, st = _run(cuda_lib, c, qkv, wq, wk, chunk_lens=True)
    assert st == 0
    q_ref, k_ref, v_ref, skipped = _oracle(c, qkv, wq, wk, chunk_lens=c.chunk_lens)
    assert skipped == 0
    _check_q(q, q_ref, "chunked q")
    _check_caches(c, cd.k_cache, cd.v_cache, k_ref, v_ref, "chunked", chunked=True)


def test_invalid_sequence_flags_and_writes_nothing(cuda_lib):
    c = W.custom_case(530, [300, 300, 5], Hq=8, Hkv=2)
    c.block_table[1, 2] = -1
    qkv, wq, wk = W.prologue_inputs(c, 530)
    q, cd, st = _run(cuda_lib, c, qkv, wq, wk)
    assert st & cuda_lib.PA_STATUS_BAD_PAGE
    q_ref, k_ref, v_ref, skipped = _oracle(c, qkv, wq, wk)
    assert skipped == 1
    assert torch.count_nonzero(q[1]) == 0
    _check_q(q, q_ref, "invalid neighbour")
    _check_caches(c, cd.k_cache, cd.v_cache, k_ref, v_ref, "invalid", skip=(1,))


def test_prologue_then_decode_matches_the_oracle_chain(cuda_lib):
    """Decode step with the fused prologue: GPU prologue -> pa_decode against the
    oracle prologue -> oracle attention, softmax scale folded into Q."""
    ctx = [1, 513, 4096, 2051, 64]
    c = W.custom_case(540, ctx, Hq=40, Hkv=8, max_pages_per_seq=32)
    qkv, wq, wk = W.prologue_inputs(c, 540)
    kw = dict(q_scale=1.0 / math.sqrt(D))
    q, cd, st = _run(cuda_lib, c, qkv, wq, wk, **kw)
    out = cuda_lib.pa_decode(q, cd.k_cache, cd.v_cache, cd.block_table, cd.context_lens, 1.0,
                             out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert st == 0
    q_ref, k_ref, v_ref, _ = _oracle(c, qkv, wq, wk, **kw)
    # the oracle attends its own prologue's outputs (Q rounded to bf16 like the GPU's input)
    qb = torch.from_numpy(q_ref).float().to(torch.bfloat16)
    ref = oracle.attention(qb, k_ref, v_ref, c.block_table, c.context_lens, None, 1.0,
                           c.Hq, c.Hkv, c.num_pages, c.max_pages_per_seq)
    assert_close(out, ref, what="prologue + decode")
