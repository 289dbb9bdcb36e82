"""pa_qk_norm_rope_write_fp8 (the prologue into an FP8 e4m3 cache) on the GPU.

Its cache bytes are defined as those of pa_qk_norm_rope_write followed by
pa_kv_write_fp8 of the rows it wrote: checked bit for bit against that GPU
pair (each half of which is checked against the oracle elsewhere).  Against
the oracle's composition of the same two steps: V codes and every untouched
byte bit for bit; K within the e4m3 rounding of the oracle's bf16 K (the GPU's
bf16 K may sit one bf16 ulp away, so a code one step over a rounding boundary
is allowed); Q as in the bf16 prologue; and the prologue -> pa_decode_fp8
chain against oracle attention over the oracle's caches."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from pa_testutil import assert_close, dev_status

pytestmark = pytest.mark.gpu
D = 128


def _scales(Hkv, seed):
    g = torch.Generator().manual_seed(seed)
    ks = (torch.rand(Hkv, generator=g) * 0.02 + 0.02).float()
    vs = (torch.rand(Hkv, generator=g) * 0.02 + 0.02).float()
    return ks, vs


def _fp8(cache, scale):
    """Starting FP8 cache (an input): the case's bf16 values over the scale."""
    return (cache.float() / scale[None, None, :, None]).to(torch.float8_e4m3fn).view(torch.uint8)


def _written(c, chunked, skip=()):
    """(token, page, offset) of every new token of a valid sequence."""
    out, tok = [], 0
    for s in range(c.B):
        ctx = int(c.context_lens[s])
        n = int(c.chunk_lens[s]) if chunked else 1
        for j in range(n):
            pos = ctx - n + j
            if s not in skip:
                out.append((tok, int(c.block_table[s, pos // 128]), pos % 128))
            tok += 1
    return out


def _setup(seed, ctx, chunk=None, Hq=8, Hkv=2, **kw):
    c = W.custom_case(seed, ctx, Hq=Hq, Hkv=Hkv, chunk_lens=chunk, **kw)
    qkv, wq, wk = W.prologue_inputs(c, seed)
    ks, vs = _scales(Hkv, seed)
    return c, qkv, wq, wk, ks, vs, _fp8(c.k_cache, ks), _fp8(c.v_cache, vs)


def _gpu_fused(pa, c, qkv, wq, wk, ks, vs, k8, v8, chunked, **kw):
    cd = c.to("cuda")
    kc, vc = k8.cuda(), v8.cuda()
    st = dev_status()
    q = pa.pa_qk_norm_rope_write_fp8(qkv.cuda(), wq.cuda(), wk.cuda(), kc, vc, ks.cuda(),
                                     vs.cuda(), cd.block_table, cd.context_lens,
                                     cd.chunk_lens if chunked else None, status=st, **kw)
    torch.cuda.synchronize()
    return q, kc, vc, int(st.item())


def _gpu_two_step(pa, c, qkv, wq, wk, ks, vs, k8, v8, chunked, **kw):
    """pa_qk_norm_rope_write into a bf16 cache, then pa_kv_write_fp8 of the rows
    it wrote (gathered from their slots, in token order)."""
    cd = c.to("cuda")
    cl = cd.chunk_lens if chunked else None
    q = pa.pa_qk_norm_rope_write(qkv.cuda(), wq.cuda(), wk.cuda(), cd.k_cache, cd.v_cache,
                                 cd.block_table, cd.context_lens, cl, **kw)
    slots = _written(c, chunked)
    pages = torch.tensor([p for _, p, _ in slots], device="cuda")
    offs = torch.tensor([o for _, _, o in slots], device="cuda")
    k_rows = cd.k_cache[pages, offs].contiguous()
    v_rows = cd.v_cache[pages, offs].contiguous()
    kc, vc = k8.cuda(), v8.cuda()
    pa.pa_kv_write_fp8(k_rows, v_rows, kc, vc, ks.cuda(), vs.cuda(), cd.block_table,
                       cd.context_lens, cl)
    torch.cuda.synchronize()
    return q, kc, vc


def _oracle(c, qkv, wq, wk, ks, vs, k8, v8, chunked, **kw):
    return oracle.qk_norm_rope_write_fp8(
        qkv, wq.numpy(), wk.numpy(), k8.numpy(), v8.numpy(), ks.numpy(), vs.numpy(),
        c.block_table, c.context_lens, c.chunk_lens if chunked else None, c.Hq, c.Hkv,
        c.num_pages, c.max_pages_per_seq, **kw)


def _check_q(q_gpu, q_ref, what):
    g = q_gpu.detach().float().cpu().double().numpy()
    scale = np.abs(q_ref).max(axis=-1, keepdims=True) + 1e-30
    err = np.abs(g - q_ref)
    bad = err > 2.0 ** -8 * np.abs(q_ref) + 2.0 ** -11 * scale
    assert not bad.any(), f"{what}: {bad.sum()} q values off, max err {err.max():.3e}"


def _check_oracle(c, kc, vc, k_ref, v_ref, k8, v8, ks, chunked, what, skip=()):
    kg, vg = kc.cpu().numpy(), vc.cpu().numpy()
    assert np.array_equal(vg, v_ref), f"{what}: V codes differ from the oracle"
    written = np.zeros(kg.shape[:2], dtype=bool)
    for _, page, off in _written(c, chunked, skip):
        written[page, off] = True
    assert np.array_equal(kg[~written], k8.numpy()[~written]), f"{what}: other K bytes changed"
    assert np.array_equal(k_ref[~written], k8.numpy()[~written])
    # K: the decoded codes of both sides, in units of the scale
    a = oracle.e4m3_decode(kg[written])
    b = oracle.e4m3_decode(k_ref[written])
    assert np.isfinite(a).all() and np.isfinite(b).all()
    # one e4m3 step of the larger magnitude (8 steps per binade; 2^-9 below 2^-6)
    step = np.maximum(2.0 ** np.floor(np.log2(np.maximum(np.abs(b), 2.0 ** -6))) / 8, 2.0 ** -9)
    diff = np.abs(a - b)
    assert np.all(diff <= step * (1 + 1e-12)), f"{what}: K codes differ by more than one step"
    frac = float((diff > 0).mean())
    assert frac < 0.01, f"{what}: {frac:.3%} of K codes off by one step"
    return frac


@pytest.mark.parametrize("hq,hkv", [(40, 8), (64, 8), (8, 1)])
def test_decode_prologue_fp8(cuda_lib, hq, hkv):
    ctx = [1, 200, 4096, 37, 129, 128]
    c, qkv, wq, wk, ks, vs, k8, v8 = _setup(900 + hq, ctx, Hq=hq, Hkv=hkv, max_pages_per_seq=32)
    kw = dict(eps=1e-6, rope_base=1e6, rope_scale=1.0, q_scale=1.0 / math.sqrt(D))
    q, kc, vc, st = _gpu_fused(cuda_lib, c, qkv, wq, wk, ks, vs, k8, v8, False, **kw)
    assert st == 0
    q2, kc2, vc2 = _gpu_two_step(cuda_lib, c, qkv, wq, wk, ks, vs, k8, v8, False, **kw)
    assert torch.equal(q, q2)
    assert torch.equal(kc, kc2) and torch.equal(vc, vc2), "fused != prologue + pa_kv_write_fp8"
    q_ref, k_ref, v_ref, skipped = _oracle(c, qkv, wq, wk, ks, vs, k8, v8, False, **kw)
    assert skipped == 0
    _check_q(q, q_ref, f"fp8 prologue q {hq}/{hkv}")
    _check_oracle(c, kc, vc, k_ref, v_ref, k8, v8, ks, False, f"decode {hq}/{hkv}")


def test_chunked_prefill_prologue_fp8_full_size(cuda_lib):
    """The benchmark's chunked prefill: 8 sequences x 512 new tokens (T = 4096)."""
    c = W.chunked_prefill()
    qkv, wq, wk = W.prologue_inputs(c, 920)
    ks, vs = _scales(c.Hkv, 920)
    k8, v8 = _fp8(c.k_cache, ks), _fp8(c.v_cache, vs)
    q, kc, vc, st = _gpu_fused(cuda_lib, c, qkv, wq, wk, ks, vs, k8, v8, True)
    assert st == 0
    q2, kc2, vc2 = _gpu_two_step(cuda_lib, c, qkv, wq, wk, ks, vs, k8, v8, True)
    assert torch.equal(q, q2) and torch.equal(kc, kc2) and torch.equal(vc, vc2)
    q_ref, k_ref, v_ref, skipped = _oracle(c, qkv, wq, wk, ks, vs, k8, v8, True)
    assert skipped == 0
    _check_q(q, q_ref, "chunked fp8 q")
    _check_oracle(c, kc, vc, k_ref, v_ref, k8, v8, ks, True, "chunked")


def test_invalid_sequence_fp8_flags_and_writes_nothing(cuda_lib):
    c, qkv, wq, wk, ks, vs, k8, v8 = _setup(930, [300, 300, 5], chunk=[2, 300, 5])
    c.block_table[1, 2] = -1
    q, kc, vc, st = _gpu_fused(cuda_lib, c, qkv, wq, wk, ks, vs, k8, v8, True)
    assert st & cuda_lib.PA_STATUS_BAD_PAGE
    q_ref, k_ref, v_ref, skipped = _oracle(c, qkv, wq, wk, ks, vs, k8, v8, True)
    assert skipped == 1
    assert torch.count_nonzero(q[2:302]) == 0
    _check_q(q, q_ref, "invalid neighbour")
    _check_oracle(c, kc, vc, k_ref, v_ref, k8, v8, ks, True, "invalid", skip=(1,))


def test_prologue_fp8_then_decode_matches_the_oracle_chain(cuda_lib):
    """Decode step over an FP8 cache with the fused prologue: GPU prologue ->
    pa_decode_fp8 against the oracle prologue -> oracle FP8 attention, the
    softmax scale folded into Q."""
    ctx = [1, 513, 4096, 2051, 64]
    c, qkv, wq, wk, ks, vs, k8, v8 = _setup(940, ctx, Hq=40, Hkv=8, max_pages_per_seq=32)
    kw = dict(q_scale=1.0 / math.sqrt(D))
    q, kc, vc, st = _gpu_fused(cuda_lib, c, qkv, wq, wk, ks, vs, k8, v8, False, **kw)
    out = cuda_lib.pa_decode_fp8(q, kc, vc, ks.cuda(), vs.cuda(), c.block_table.cuda(),
                                 c.context_lens.cuda(), 1, 1.0, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert st == 0
    q_ref, k_ref, v_ref, _ = _oracle(c, qkv, wq, wk, ks, vs, k8, v8, False, **kw)
    qb = torch.from_numpy(q_ref).float().to(torch.bfloat16)
    ref = oracle.attention_fp8(qb, k_ref, v_ref, ks.numpy(), vs.numpy(), c.block_table,
                               c.context_lens, None, 1.0, c.Hq, c.Hkv, c.num_pages,
                               c.max_pages_per_seq)
    assert_close(out, ref, what="fp8 prologue + decode")
