"""Pins for the FP64 oracle: each checks it against something other than itself
(closed forms, invariants, a textbook routine, brute force on tiny inputs)."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
D, P = W.HEAD_DIM, W.PAGE


def _bf(x):
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16)


def _f64(t):
    return t.float().double().numpy()


def _attn(c, rows=None, scale=None, chunk=True):
    return oracle.attention(c.q, c.k_cache, c.v_cache, c.block_table, c.context_lens,
                            c.chunk_lens if chunk else None, c.scale if scale is None else scale,
                            c.Hq, c.Hkv, c.num_pages, c.max_pages_per_seq, rows=rows)


def _golden(name):
    vals = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split()
            vals[k] = float(v)
    return vals


def test_golden_two_key_closed_form():
    g = _golden("two_token_softmax.txt")
    kc = torch.zeros(3, P, 1, D, dtype=torch.bfloat16)
    vc = torch.zeros(3, P, 1, D, dtype=torch.bfloat16)
    kc[0].fill_(float("nan")); vc[0].fill_(float("nan"))   # unreferenced pages
    kc[1].fill_(float("nan")); vc[1].fill_(float("nan"))
    kc[2, 2:].fill_(float("nan")); vc[2, 2:].fill_(float("nan"))  # tail slots
    kc[2, 1, 0, 0] = 2.0
    vc[2, 0, 0, 0] = 1.0
    vc[2, 1, 0, 1] = 1.0
    q = torch.zeros(1, 1, D, dtype=torch.bfloat16)
    q[0, 0, 0] = 1.0
    out = oracle.attention(q, kc, vc, torch.tensor([[2]], dtype=torch.int32),
                           torch.tensor([2], dtype=torch.int32), None, 0.5, 1, 1, 3, 1)
    assert out.shape == (1, 1, D)
    assert abs(out[0, 0, 0] - g["out0"]) < 1e-15
    assert abs(out[0, 0, 1] - g["out1"]) < 1e-15
    assert np.all(out[0, 0, 2:] == 0.0)
    # the dense step's normaliser
    o, lse = oracle.dense_attention(_f64(q[0, 0]), np.stack([np.zeros(D), 2 * np.eye(D)[0]]),
                                    np.stack([np.eye(D)[0], np.eye(D)[1]]), 0.5)
    assert abs(lse - g["lse"]) < 1e-15 and abs(o[1] - g["out1"]) < 1e-15


def test_single_token_context_returns_v_exactly():
    c = W.custom_case(101, [1, 1, 1], Hq=8, Hkv=2)
    out = _attn(c)
    for s in range(3):
        page = int(c.block_table[s, 0])
        for g in range(8):
            v = _f64(c.v_cache[page, 0, g // 4])
            assert np.array_equal(out[s, g], v)


def test_identical_keys_give_mean_of_v():
    c = W.custom_case(102, [77, 300], Hq=4, Hkv=1)
    c.k_cache[:] = _bf(torch.randn(D, generator=torch.Generator().manual_seed(9)))  # every key identical
    out = _attn(c)
    for s, n in enumerate([77, 300]):
        vs = np.stack([_f64(c.v_cache[int(c.block_table[s, t // P]), t % P, 0]) for t in range(n)])
        np.testing.assert_allclose(out[s, :], np.broadcast_to(vs.mean(0), (4, D)), rtol=0, atol=1e-12)


def test_zero_scale_gives_mean_of_v():
    c = W.custom_case(103, [129], Hq=2, Hkv=1)
    out = _attn(c, scale=0.0)
    vs = np.stack([_f64(c.v_cache[int(c.block_table[0, t // P]), t % P, 0]) for t in range(129)])
    np.testing.assert_allclose(out[0], np.broadcast_to(vs.mean(0), (2, D)), atol=1e-12, rtol=0)


def test_constant_v_rows_give_that_constant():
    c = W.custom_case(104, [250, 5], Hq=6, Hkv=3)
    cval = _bf(torch.randn(3, D, generator=torch.Generator().manual_seed(7)))
    for h in range(3):
        c.v_cache[:, :, h, :] = cval[h]
    out = _attn(c)
    for g in range(6):
        np.testing.assert_allclose(out[:, g], np.broadcast_to(_f64(cval[g // 2]), (2, D)), atol=1e-12, rtol=0)


def test_empty_context_is_zero_and_others_unaffected():
    c = W.custom_case(105, [0, 40], Hq=4, Hkv=2)
    out = _attn(c)
    assert np.all(out[0] == 0.0)
    c2 = W.custom_case(105, [0, 40], Hq=4, Hkv=2)
    c2.context_lens = torch.tensor([0, 40], dtype=torch.int32)
    assert np.isfinite(out[1]).all() and np.abs(out[1]).sum() > 0


def test_linearity_in_v():
    rng = np.random.default_rng(11)
    c = W.custom_case(106, [200, 64], Hq=4, Hkv=2)
    v1 = torch.as_tensor(rng.integers(-32, 33, size=c.v_cache.shape), dtype=torch.float32).to(torch.bfloat16)
    v2 = torch.as_tensor(rng.integers(-32, 33, size=c.v_cache.shape), dtype=torch.float32).to(torch.bfloat16)
    outs = []
    for v in (v1, v2, (v1.float() + v2.float()).to(torch.bfloat16)):
        c.v_cache = v
        outs.append(_attn(c))
    np.testing.assert_allclose(outs[2], outs[0] + outs[1], atol=1e-11, rtol=0)


def test_page_permutation_is_invisible():
    c = W.custom_case(107, [300, 129, 1], Hq=8, Hkv=2, extra_pages=4)
    base = _attn(c)
    perm = torch.randperm(c.num_pages, generator=torch.Generator().manual_seed(3))
    inv = torch.empty_like(perm); inv[perm] = torch.arange(c.num_pages)
    kc, vc = c.k_cache[perm], c.v_cache[perm]          # new page i holds old page perm[i]
    bt = c.block_table.clone()
    bt[bt >= 0] = inv[bt[bt >= 0].long()].to(torch.int32)
    c.k_cache, c.v_cache, c.block_table = kc, vc, bt
    assert np.array_equal(_attn(c), base)


def test_gqa_equals_mha_with_repeated_kv_heads():
    c = W.custom_case(108, [190, 33], Hq=8, Hkv=2)
    gqa = _attn(c)
    c.k_cache = c.k_cache.repeat_interleave(4, dim=2)
    c.v_cache = c.v_cache.repeat_interleave(4, dim=2)
    c.Hkv = 8
    assert np.array_equal(_attn(c), gqa)


def _dense_case(seed, ctx_lens, chunk_lens, Hq, Hkv):
    """Build dense per-sequence K/V first, then lay them into shuffled pages."""
    g = torch.Generator().manual_seed(seed)
    B = len(ctx_lens)
    dense_k = [torch.randn(n, Hkv, D, generator=g).to(torch.bfloat16) for n in ctx_lens]
    dense_v = [torch.randn(n, Hkv, D, generator=g).to(torch.bfloat16) for n in ctx_lens]
    need = [(n + P - 1) // P for n in ctx_lens]
    npages = sum(need) + 2
    perm = torch.randperm(npages, generator=g).tolist()
    kc = torch.full((npages, P, Hkv, D), float("nan"), dtype=torch.bfloat16)
    vc = kc.clone()
    mp = max(need)
    bt = torch.full((B, mp), -1, dtype=torch.int32)
    i = 0
    for s in range(B):
        for pi in range(need[s]):
            page = perm[i]; i += 1
            bt[s, pi] = page
            lo, hi = pi * P, min(ctx_lens[s], (pi + 1) * P)
            kc[page, :hi - lo] = dense_k[s][lo:hi]
            vc[page, :hi - lo] = dense_v[s][lo:hi]
    T = sum(chunk_lens)
    q = torch.randn(T, Hq, D, generator=g).to(torch.bfloat16)
    return q, kc, vc, bt, dense_k, dense_v, npages, mp


@pytest.mark.parametrize("Hq,Hkv", [(4, 2), (6, 1), (3, 3)])
def test_matches_torch_sdpa_brute_force(Hq, Hkv):
    ctx = [5, 130, 257]
    chunk = [2, 3, 4]
    scale = 0.37
    q, kc, vc, bt, dk, dv, npages, mp = _dense_case(200 + Hq, ctx, chunk, Hq, Hkv)
    out = oracle.attention(q, kc, vc, bt, torch.tensor(ctx, dtype=torch.int32),
                           torch.tensor(chunk, dtype=torch.int32), scale, Hq, Hkv, npages, mp)
    tok = 0
    for s in range(3):
        n, c = chunk[s], ctx[s]
        qq = q[tok:tok + n].double().permute(1, 0, 2).unsqueeze(0)           # [1, Hq, n, D]
        kk = dk[s].double().permute(1, 0, 2).repeat_interleave(Hq // Hkv, 0).unsqueeze(0)
        vv = dv[s].double().permute(1, 0, 2).repeat_interleave(Hq // Hkv, 0).unsqueeze(0)
        pos = torch.arange(c - n, c).unsqueeze(1)
        mask = torch.arange(c).unsqueeze(0) <= pos                            # [n, c]
        ref = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask, scale=scale)
        np.testing.assert_allclose(out[tok:tok + n], ref[0].permute(1, 0, 2).numpy(), atol=1e-12, rtol=0)
        tok += n


def test_shared_prefix_pages_give_equal_outputs():
    c = W.custom_case(109, [300, 300], Hq=4, Hkv=2)
    c.block_table[1] = c.block_table[0]        # both sequences map the same pages
    c.q[1] = c.q[0]
    out = _attn(c)
    assert np.array_equal(out[0], out[1])


def test_prefill_single_token_equals_decode_and_last_row_equals_decode():
    c = W.custom_case(110, [200, 77], Hq=4, Hkv=2, chunk_lens=[1, 1])
    pre = _attn(c)
    dec = _attn(c, chunk=False)
    assert np.array_equal(pre, dec)
    c = W.custom_case(111, [300, 140], Hq=4, Hkv=2, chunk_lens=[20, 7])
    pre = _attn(c)
    last = torch.stack([c.q[19], c.q[26]])
    dec = oracle.attention(last, c.k_cache, c.v_cache, c.block_table, c.context_lens, None,
                           c.scale, 4, 2, c.num_pages, c.max_pages_per_seq)
    assert np.array_equal(pre[[19, 26]], dec)


def test_chunk_split_in_two_calls_equals_one_call():
    full = W.custom_case(112, [600], Hq=4, Hkv=1, chunk_lens=[512], with_new=True)
    kc, vc, sk = oracle.kv_write(full.k_new, full.v_new, full.k_cache, full.v_cache,
                                 full.block_table, full.context_lens, full.chunk_lens,
                                 full.num_pages, full.max_pages_per_seq)
    assert sk == 0
    one = oracle.attention(full.q, kc, vc, full.block_table, full.context_lens, full.chunk_lens,
                           full.scale, 4, 1, full.num_pages, full.max_pages_per_seq)
    kc2, vc2 = full.k_cache, full.v_cache
    outs = []
    for lo, hi in ((0, 256), (256, 512)):
        ctx = torch.tensor([600 - 512 + hi], dtype=torch.int32)
        n = torch.tensor([hi - lo], dtype=torch.int32)
        kc2, vc2, sk = oracle.kv_write(full.k_new[lo:hi], full.v_new[lo:hi], kc2, vc2,
                                       full.block_table, ctx, n, full.num_pages, full.max_pages_per_seq)
        assert sk == 0
        outs.append(oracle.attention(full.q[lo:hi], kc2, vc2, full.block_table, ctx, n, full.scale,
                                     4, 1, full.num_pages, full.max_pages_per_seq))
    assert np.array_equal(np.concatenate(outs), one)


def test_kv_write_round_trip_and_untouched_bytes():
    c = W.custom_case(113, [130, 1, 257], Hq=4, Hkv=2, chunk_lens=[3, 1, 129], with_new=True)
    kc, vc, sk = oracle.kv_write(c.k_new, c.v_new, c.k_cache, c.v_cache, c.block_table,
                                 c.context_lens, c.chunk_lens, c.num_pages, c.max_pages_per_seq)
    assert sk == 0
    k0 = c.k_cache.view(torch.int16).numpy().view(np.uint16)
    written = np.zeros(kc.shape[:2], dtype=bool)
    tok = 0
    for s, (ctx, n) in enumerate(zip([130, 1, 257], [3, 1, 129])):
        for j in range(n):
            pos = ctx - n + j
            page = int(c.block_table[s, pos // P])
            assert np.array_equal(kc[page, pos % P], c.k_new[tok].view(torch.int16).numpy().view(np.uint16))
            assert np.array_equal(vc[page, pos % P], c.v_new[tok].view(torch.int16).numpy().view(np.uint16))
            written[page, pos % P] = True
            tok += 1
    assert np.array_equal(kc[~written], k0[~written])      # every other byte unchanged
    assert written.sum() == c.T


def test_kv_write_skips_invalid_sequence():
    c = W.custom_case(114, [10, 10], Hq=2, Hkv=1, chunk_lens=[2, 2], with_new=True)
    c.block_table[1, 0] = c.num_pages          # out of range
    kc, vc, sk = oracle.kv_write(c.k_new, c.v_new, c.k_cache, c.v_cache, c.block_table,
                                 c.context_lens, c.chunk_lens, c.num_pages, c.max_pages_per_seq)
    assert sk == 1
    page0 = int(c.block_table[0, 0])
    assert np.array_equal(kc[page0, 8], c.k_new[0].view(torch.int16).numpy().view(np.uint16))


def test_invalid_page_zeroes_only_that_sequence():
    c = W.custom_case(115, [200, 200], Hq=4, Hkv=2)
    good = _attn(c)
    c.block_table[0, 1] = -1
    out = _attn(c)
    assert np.all(out[0] == 0.0)
    assert np.array_equal(out[1], good[1])


def test_poison_never_leaks():
    c = W.tiny_decode()
    out = _attn(c)
    assert np.isfinite(out).all()
    c = W.custom_case(116, [1, 63, 64, 65, 127, 128, 129], Hq=4, Hkv=1)
    assert np.isfinite(_attn(c)).all()


def test_combine_of_key_ranges_equals_full_attention():
    rng = np.random.default_rng(5)
    n = 700
    q = rng.standard_normal(D)
    K = rng.standard_normal((n, D))
    V = rng.standard_normal((n, D))
    full, full_lse = oracle.dense_attention(q, K, V, 0.09)
    cuts = [0, 1, 128, 300, 300, 699, 700]     # includes an empty range
    po, pl = [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        o, l = oracle.dense_attention(q, K[a:b], V[a:b], 0.09)
        po.append(o); pl.append(l)
    assert pl[3] == -math.inf
    merged = oracle.combine(np.array(po)[None], np.array(pl)[None])
    np.testing.assert_allclose(merged[0], full, atol=1e-13, rtol=0)
    # all-empty row merges to zero
    z = oracle.combine(np.zeros((1, 2, D)), np.full((1, 2), -np.inf))
    assert np.all(z == 0.0)


def test_five_workloads_build_and_fit():
    c = W.tiny_decode()
    assert c.B == 2 and c.Hq == 8 and c.Hkv == 2 and c.num_pages == 4 and c.poisoned_pages
    c = W.qwen3_14b_decode_b16()
    assert c.B == 16 and c.Hq == 40 and c.Hkv == 8 and c.num_pages == 512
    c = W.chunked_prefill()
    assert c.T == 4096 and int(c.context_lens.max()) <= 4096
