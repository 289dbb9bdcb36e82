"""Pins for the oracle's FP8 KV cache (an "fp8_e4m3" KV cache, as in the SGLang
measurement quoted by the "Qwen4-Exp QSA trafia na Ascend..." blog; a
quantized KV dtype is also the --kv-cache-dtype option of the "Qwen 3"
TensorSharp doc, section 11).  The e4m3 codec is pinned to torch's
float8_e4m3fn conversions (a library routine) and to closed forms; the FP8
KV write and attention are pinned to the bf16 oracle through exact
power-of-two scales and to the scale identities of the softmax."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W

CODES = np.arange(256, dtype=np.uint8)


def _torch_decode(codes):
    return torch.from_numpy(np.asarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn) \
        .to(torch.float64).numpy()


def _torch_encode(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn) \
        .view(torch.uint8).numpy()


def test_decode_every_code_matches_float8_e4m3fn():
    mine, ref = oracle.e4m3_decode(CODES), _torch_decode(CODES)
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    assert np.array_equal(mine[~np.isnan(mine)], ref[~np.isnan(ref)])
    assert np.isnan(mine).sum() == 2 and np.isnan(mine[[0x7F, 0xFF]]).all()
    assert mine[0x7E] == 448.0 and mine[0x01] == 2.0 ** -9 and mine[0x08] == 2.0 ** -6


def test_encode_in_range_matches_float8_e4m3fn():
    rng = np.random.default_rng(7)
    finite = oracle.e4m3_decode(CODES[:0x7F])          # 0 .. 448
    mids = (finite[:-1] + finite[1:]) / 2               # every tie between neighbours
    x = np.concatenate([rng.uniform(-448, 448, 50000), rng.normal(0, 0.02, 50000),
                        finite, -finite, mids, -mids,
                        np.nextafter(mids.astype(np.float32), np.float32(np.inf)),
                        np.nextafter(mids.astype(np.float32), np.float32(-np.inf))])
    x = x.astype(np.float32)
    x = x[np.abs(x) <= 448]
    assert np.array_equal(oracle.e4m3_encode(x), _torch_encode(x))


def test_encode_closed_forms():
    enc = lambda v: int(oracle.e4m3_encode(np.array([v], dtype=np.float32))[0])
    assert enc(448.0) == 0x7E and enc(449.0) == 0x7E and enc(1e30) == 0x7E
    assert enc(np.inf) == 0x7E and enc(-np.inf) == 0xFE and enc(-500.0) == 0xFE
    assert enc(np.nan) & 0x7F == 0x7F
    assert enc(0.0) == 0x00 and enc(-0.0) == 0x80
    assert enc(2.0 ** -10) == 0x00            # half the least subnormal: tie -> even 0
    assert enc(3 * 2.0 ** -10) == 0x02        # between 2^-9 (odd) and 2^-8 (even)
    assert enc(1.0 + 1 / 16) == 0x38          # between 1 (even) and 1.125: 1
    assert enc(1.0 + 3 / 16) == 0x3A          # between 1.125 and 1.25 (even): 1.25
    assert enc(2.0 ** -20) == 0x00 and enc(-(2.0 ** -20)) == 0x80


def test_round_trip_of_every_finite_code():
    fin = CODES[~np.isnan(oracle.e4m3_decode(CODES))]
    back = oracle.e4m3_encode(oracle.e4m3_decode(fin).astype(np.float32))
    # +0 and -0 are distinct codes and both round-trip
    assert np.array_equal(back, fin)


def _fp8_case(seed, ctx, chunk, Hq=8, Hkv=2):
    case = W.custom_case(seed, ctx, Hq=Hq, Hkv=Hkv, chunk_lens=chunk, with_new=True)
    rng = np.random.default_rng(seed)
    kc = rng.integers(0, 256, size=case.k_cache.shape, dtype=np.uint8)
    vc = rng.integers(0, 256, size=case.v_cache.shape, dtype=np.uint8)
    for c in (kc, vc):                       # no NaN codes in the prior context
        c[(c & 0x7F) == 0x7F] = 0x3C
    return case, kc, vc


def test_kv_write_fp8_quantizes_into_the_slots():
    case, kc, vc = _fp8_case(31, [130, 300], [3, 129])
    ks = np.array([0.5, 0.03125], dtype=np.float32)
    vs = np.array([0.75, 3.0], dtype=np.float32)
    k2, v2, skipped = oracle.kv_write_fp8(case.k_new, case.v_new, kc, vc, ks, vs,
                                          case.block_table, case.context_lens, case.chunk_lens,
                                          case.num_pages, case.max_pages_per_seq)
    assert skipped == 0
    rowsk = np.asarray(case.k_new.float() / torch.from_numpy(ks)[None, :, None])
    rowsv = np.asarray(case.v_new.float() / torch.from_numpy(vs)[None, :, None])
    bt = case.block_table.numpy()
    tok, written = 0, np.zeros(kc.shape[:2], dtype=bool)
    for s, (c, n) in enumerate(zip(case.context_lens.tolist(), case.chunk_lens.tolist())):
        for j in range(n):
            pos = c - n + j
            page, off = bt[s, pos // 128], pos % 128
            assert np.array_equal(k2[page, off], oracle.e4m3_encode(rowsk[tok]))
            assert np.array_equal(v2[page, off], oracle.e4m3_encode(rowsv[tok]))
            inr = np.abs(rowsk[tok]) <= 448
            assert np.array_equal(k2[page, off][inr], _torch_encode(rowsk[tok][inr]))
            written[page, off] = True
            tok += 1
    assert np.array_equal(k2[~written], kc[~written]) and np.array_equal(v2[~written], vc[~written])


def test_kv_write_fp8_skips_an_invalid_sequence():
    case, kc, vc = _fp8_case(32, [200, 100], [4, 4])
    last = int(case.block_table[1, 0])        # sequence 1's only page (positions 96..99)
    case.block_table[1, 0] = case.num_pages + 5
    ones = np.ones(2, dtype=np.float32)
    k2, v2, skipped = oracle.kv_write_fp8(case.k_new, case.v_new, kc, vc, ones, ones,
                                          case.block_table, case.context_lens, case.chunk_lens,
                                          case.num_pages, case.max_pages_per_seq)
    assert skipped == 1
    assert np.array_equal(k2[last], kc[last]) and np.array_equal(v2[last], vc[last])
    p0 = int(case.block_table[0, 1])          # sequence 0 (positions 196..199) was written
    assert not np.array_equal(k2[p0, 68:72], kc[p0, 68:72])


def _bf16_of(values):
    return torch.from_numpy(values.astype(np.float32)).to(torch.bfloat16)


def test_attention_fp8_equals_bf16_oracle_under_power_of_two_scales():
    """With power-of-two scales every dequantized value is exactly a bf16, so the
    FP8 attention must equal the bf16 oracle on the dequantized cache bit for bit."""
    case, kc, vc = _fp8_case(33, [700, 129, 5], [3, 129, 5])
    ks = np.array([0.25, 2.0], dtype=np.float32)
    vs = np.array([0.5, 0.125], dtype=np.float32)
    kd = oracle.e4m3_decode(kc) * ks[None, None, :, None]
    vd = oracle.e4m3_decode(vc) * vs[None, None, :, None]
    a = oracle.attention_fp8(case.q, kc, vc, ks, vs, case.block_table, case.context_lens,
                             case.chunk_lens, case.scale, case.Hq, case.Hkv, case.num_pages,
                             case.max_pages_per_seq)
    b = oracle.attention(case.q, _bf16_of(kd), _bf16_of(vd), case.block_table,
                         case.context_lens, case.chunk_lens, case.scale, case.Hq, case.Hkv,
                         case.num_pages, case.max_pages_per_seq)
    assert np.array_equal(a, b)


def test_attention_fp8_scale_identities():
    """k_scale multiplies every score of its KV head (the same as scaling the
    softmax scale); v_scale multiplies the output of its KV head."""
    case, kc, vc = _fp8_case(34, [300, 40], None)
    ones = np.ones(2, dtype=np.float32)
    ks = np.array([0.037, 1.9], dtype=np.float32)
    vs = np.array([0.61, 0.0173], dtype=np.float32)
    args = (case.block_table, case.context_lens, None)
    base = oracle.attention_fp8(case.q, kc, vc, ones, ones, *args, case.scale, case.Hq,
                                case.Hkv, case.num_pages, case.max_pages_per_seq)
    got = oracle.attention_fp8(case.q, kc, vc, ks, vs, *args, case.scale, case.Hq, case.Hkv,
                               case.num_pages, case.max_pages_per_seq)
    G = case.Hq // case.Hkv
    for h in range(case.Hkv):
        hs = slice(h * G, (h + 1) * G)
        ref = oracle.attention_fp8(case.q, kc, vc, ones, ones, *args,
                                   case.scale * float(ks[h]), case.Hq, case.Hkv,
                                   case.num_pages, case.max_pages_per_seq)
        np.testing.assert_allclose(got[:, hs], float(vs[h]) * ref[:, hs], rtol=1e-12,
                                   atol=1e-14)
    assert not np.allclose(got, base)


# ---- the prologue over an FP8 cache: the bf16 prologue's rows, quantized

def _bits_f32(b):
    return (np.asarray(b, dtype=np.uint32) << 16).view(np.float32)


def _prologue_fp8_case(seed, ctx, chunk_lens=None, hq=8, hkv=2):
    c = W.custom_case(seed, ctx, Hq=hq, Hkv=hkv, chunk_lens=chunk_lens)
    qkv, wq, wk = W.prologue_inputs(c, seed)
    g = np.random.default_rng(seed)
    ks = (g.random(hkv) * 0.02 + 0.02).astype(np.float32)
    vs = (g.random(hkv) * 0.02 + 0.02).astype(np.float32)
    k8 = np.full(tuple(c.k_cache.shape), 0x5A, dtype=np.uint8)   # untouched-byte markers
    v8 = np.full(tuple(c.v_cache.shape), 0xA5, dtype=np.uint8)
    return c, qkv, wq.numpy(), wk.numpy(), ks, vs, k8, v8


def _slots(c, chunk_lens, skip=()):
    """(token index, page, offset) of the new tokens of valid sequences."""
    out, tok = [], 0
    for s in range(c.B):
        n = 1 if chunk_lens is None else int(chunk_lens[s])
        ctx = int(c.context_lens[s])
        for j in range(n):
            pos = ctx - n + j
            if s not in skip:
                out.append((tok, int(c.block_table[s, pos // 128]), pos % 128))
            tok += 1
    return out


@pytest.mark.parametrize("ctx,chunk,bad", [([1, 200, 129], None, None),
                                           ([300, 260, 5], [3, 130, 5], 1)])
def test_prologue_fp8_quantizes_the_bf16_prologue_rows(ctx, chunk, bad):
    c, qkv, wq, wk, ks, vs, k8, v8 = _prologue_fp8_case(611 + len(ctx), ctx, chunk)
    if bad is not None:
        c.block_table[bad, 1] = -1
    cl = None if chunk is None else np.array(chunk, dtype=np.int32)
    args = (c.block_table, c.context_lens, cl, c.Hq, c.Hkv, c.num_pages, c.max_pages_per_seq)
    q8, kc8, vc8, sk8 = oracle.qk_norm_rope_write_fp8(qkv, wq, wk, k8, v8, ks, vs, *args)
    q, kc, _, sk = oracle.qk_norm_rope_write(qkv, wq, wk, c.k_cache, c.v_cache, *args)
    assert sk8 == sk == (0 if bad is None else 1)
    assert np.array_equal(q8, q)
    x = oracle._u16(qkv).reshape(c.T, c.Hq + 2 * c.Hkv, 128)
    written = np.zeros(kc8.shape[:2], dtype=bool)
    slots = _slots(c, chunk, skip=() if bad is None else (bad,))
    assert slots
    for tok, page, off in slots:
        written[page, off] = True
        # K: the bf16 prologue's row over k_scale (an FP32 quotient), then e4m3 by
        # torch's float8_e4m3fn conversion
        assert np.array_equal(kc8[page, off], _torch_encode(_bits_f32(kc[page, off]) / ks[:, None]))
        # V: the input row over v_scale
        v_in = _bits_f32(x[tok, c.Hq + c.Hkv:])
        assert np.array_equal(vc8[page, off], _torch_encode(v_in / vs[:, None]))
    # no other byte changes (an invalid sequence writes nothing)
    assert np.all(kc8[~written] == 0x5A) and np.all(vc8[~written] == 0xA5)
