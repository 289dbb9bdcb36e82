"""Pins for the oracle's decode/prefill prologue (Q/K RMSNorm -> NeoX RoPE ->
KV cache write; "Qwen 3" TensorSharp doc, sections 3, 4.1, 4.3, 5; "Qwen3-14B"
pypto-lib doc, "Model structure, top down").  Each test checks the oracle
against something the pages or the mathematics fix: closed forms at special
bases and positions, rotation invariants, RMSNorm identities, and where the
K/V rows land."""
import numpy as np
import pytest

import oracle
import workloads as W

D = 128
rng = np.random.default_rng(1234)


def _bf16_bits(x):
    """float array -> bf16 bit patterns (round to nearest even), for test inputs."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def _bits_to_f64(b):
    return (np.asarray(b, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


# ---- RoPE (section 4.1: NeoX style, frequencies from freq_base and scale)

def test_rope_position_zero_is_identity():
    x = rng.standard_normal(D)
    assert np.array_equal(oracle.rope_neox(x, 0.0, 1e6), x)


@pytest.mark.parametrize("scale", [1.0, 2.0, 8.0])
def test_rope_base_one_rotates_every_pair_by_pos_over_scale(scale):
    # base 1: every frequency is 1/scale, so pair (i, i+64) turns by pos/scale
    pos = 37.0
    for i in (0, 17, 63):
        e = np.zeros(D); e[i] = 1.0
        y = oracle.rope_neox(e, pos, 1.0, scale)
        assert y[i] == pytest.approx(np.cos(pos / scale), abs=1e-15)
        assert y[i + 64] == pytest.approx(np.sin(pos / scale), abs=1e-15)
        e2 = np.zeros(D); e2[i + 64] = 1.0
        y2 = oracle.rope_neox(e2, pos, 1.0, scale)
        assert y2[i] == pytest.approx(-np.sin(pos / scale), abs=1e-15)
        assert y2[i + 64] == pytest.approx(np.cos(pos / scale), abs=1e-15)


def test_rope_base_two_to_the_64_halves_the_frequency_per_pair():
    # base 2^(D/2): f_i = 2^(-i) exactly
    pos = 1000.0
    for i in (0, 1, 5, 30):
        e = np.zeros(D); e[i] = 1.0
        y = oracle.rope_neox(e, pos, 2.0 ** 64)
        assert y[i] == pytest.approx(np.cos(pos * 2.0 ** -i), abs=1e-12)
        assert y[i + 64] == pytest.approx(np.sin(pos * 2.0 ** -i), abs=1e-12)
        others = np.delete(y, [i, i + 64])
        assert np.all(others == 0.0)


def test_rope_preserves_each_pair_norm():
    x = rng.standard_normal(D)
    y = oracle.rope_neox(x, 4093.0, 1e6)
    np.testing.assert_allclose(np.hypot(y[:64], y[64:]), np.hypot(x[:64], x[64:]), rtol=1e-13)


def test_rope_scores_depend_only_on_relative_position():
    q, k = rng.standard_normal(D), rng.standard_normal(D)
    a = oracle.rope_neox(q, 100.0, 1e6) @ oracle.rope_neox(k, 37.0, 1e6)
    b = oracle.rope_neox(q, 3163.0, 1e6) @ oracle.rope_neox(k, 3100.0, 1e6)
    assert a == pytest.approx(b, rel=1e-11)


def test_rope_composes_additively():
    x = rng.standard_normal(D)
    twice = oracle.rope_neox(oracle.rope_neox(x, 300.0, 1e6), 77.0, 1e6)
    np.testing.assert_allclose(twice, oracle.rope_neox(x, 377.0, 1e6), atol=1e-12)


# ---- the whole prologue on small caches

def _case(ctx_lens, hq=4, hkv=2, chunk_lens=None, seed=7):
    c = W.custom_case(seed, ctx_lens, Hq=hq, Hkv=hkv, chunk_lens=chunk_lens, with_new=False)
    T = len(ctx_lens) if chunk_lens is None else int(sum(chunk_lens))
    return c, T


def _run(c, qkv_bits, wq, wk, chunk_lens=None, **kw):
    return oracle.qk_norm_rope_write(qkv_bits, wq, wk, c.k_cache, c.v_cache, c.block_table,
                                     c.context_lens, chunk_lens, c.Hq, c.Hkv, c.num_pages,
                                     c.max_pages_per_seq, **kw)


def test_rmsnorm_gives_unit_rms_at_position_zero():
    # ctx = 1: the new token sits at position 0, where RoPE is the identity
    c, T = _case([1, 1])
    x = rng.standard_normal((T, (c.Hq + 2 * c.Hkv) * D)) * 3.0
    q, kc, vc, skipped = _run(c, _bf16_bits(x), np.ones(D), np.ones(D), eps=0.0)
    assert skipped == 0
    np.testing.assert_allclose(np.sqrt((q ** 2).mean(-1)), 1.0, rtol=1e-13)
    xb = _bits_to_f64(_bf16_bits(x)).reshape(T, -1, D)
    ref = xb[:, :c.Hq] / np.sqrt((xb[:, :c.Hq] ** 2).mean(-1, keepdims=True))
    np.testing.assert_allclose(q, ref, rtol=1e-13)


def test_rmsnorm_is_scale_invariant_and_applies_weights_and_eps():
    c, T = _case([1, 1])
    x = rng.standard_normal((T, (c.Hq + 2 * c.Hkv) * D))
    w = rng.uniform(0.5, 1.5, D).astype(np.float32)
    q1 = _run(c, _bf16_bits(x), w, w, eps=0.0)[0]
    q2 = _run(c, _bf16_bits(4.0 * x), w, w, eps=0.0)[0]     # x4 is exact in bf16
    np.testing.assert_allclose(q1, q2, rtol=1e-14)
    q3 = _run(c, _bf16_bits(x), np.ones(D), np.ones(D), eps=0.0)[0]
    np.testing.assert_allclose(q1, q3 * w.astype(np.float64), rtol=1e-14)
    # constant head c: y = c / sqrt(c^2 + eps)
    xc = np.full((T, (c.Hq + 2 * c.Hkv) * D), 0.0078125)  # 2^-7
    q4 = _run(c, _bf16_bits(xc), np.ones(D), np.ones(D), eps=1e-4)[0]
    np.testing.assert_allclose(q4, 0.0078125 / np.sqrt(0.0078125 ** 2 + 1e-4), rtol=1e-13)


def test_q_scale_multiplies_q_only():
    c, T = _case([1, 300])
    x = rng.standard_normal((T, (c.Hq + 2 * c.Hkv) * D))
    q1, k1, v1, _ = _run(c, _bf16_bits(x), np.ones(D), np.ones(D))
    q2, k2, v2, _ = _run(c, _bf16_bits(x), np.ones(D), np.ones(D), q_scale=0.125)
    np.testing.assert_allclose(q2, 0.125 * q1, rtol=1e-15)
    assert np.array_equal(k1, k2) and np.array_equal(v1, v2)


def test_kv_rows_land_at_the_slot_with_k_normed_and_v_copied():
    c, T = _case([1, 130], hq=4, hkv=2)
    x = np.zeros((T, (c.Hq + 2 * c.Hkv), D))
    # K head h of token t is the constant (t + 1) * (h + 1) / 8; V heads random
    for t in range(T):
        for h in range(c.Hkv):
            x[t, c.Hq + h] = (t + 1) * (h + 1) / 8.0
    x[:, c.Hq + c.Hkv:] = rng.standard_normal((T, c.Hkv, D))
    bits = _bf16_bits(x.reshape(T, -1))
    q, kc, vc, skipped = _run(c, bits, np.ones(D), np.ones(D), eps=0.0)
    assert skipped == 0
    k0, v0 = oracle._u16(c.k_cache), oracle._u16(c.v_cache)
    changed_k = np.argwhere((kc != k0).any(-1))
    slots = []
    for s in range(2):
        pos = int(c.context_lens[s]) - 1
        page = int(c.block_table[s, pos // 128])
        slots.append((page, pos % 128))
        v_row = bits.reshape(T, -1, D)[s, c.Hq + c.Hkv:]
        assert np.array_equal(vc[page, pos % 128], v_row)
    # only those two slots changed, in both caches
    assert {(int(a), int(b)) for a, b, _ in changed_k} == set(slots)
    assert {(int(a), int(b)) for a, b, _ in np.argwhere((vc != v0).any(-1))} <= set(slots)
    # sequence 0 is at position 0 (no rotation): a constant head normalises to exactly 1.0
    page, off = slots[0]
    assert np.all(kc[page, off] == 0x3F80)
    # sequence 1 at position 129: each pair (1, 1) is rotated, norm sqrt(2)
    page, off = slots[1]
    kr = _bits_to_f64(kc[page, off])
    np.testing.assert_allclose(np.hypot(kr[:, :64], kr[:, 64:]), np.sqrt(2.0), rtol=2 ** -7)


def test_chunked_positions_follow_the_kv_write_reading():
    # a chunk of 3 new tokens at the end of a 5-token context: positions 2, 3, 4
    c, T = _case([5], hq=2, hkv=1, chunk_lens=[3])
    x = rng.standard_normal((T, (c.Hq + 2 * c.Hkv) * D))
    q, _, _, _ = _run(c, _bf16_bits(x), np.ones(D), np.ones(D), chunk_lens=np.array([3]), eps=0.0)
    xb = _bits_to_f64(_bf16_bits(x)).reshape(T, -1, D)
    for j in range(3):
        y = xb[j, 0] / np.sqrt((xb[j, 0] ** 2).mean())
        np.testing.assert_allclose(q[j, 0], oracle.rope_neox(y, 2 + j, 1e6), rtol=1e-13)


def test_invalid_sequence_is_skipped_and_its_q_zeroed():
    c, T = _case([200, 200])
    c.block_table[0, 1] = -1
    x = rng.standard_normal((T, (c.Hq + 2 * c.Hkv) * D))
    q, kc, vc, skipped = _run(c, _bf16_bits(x), np.ones(D), np.ones(D))
    assert skipped == 1
    assert np.all(q[0] == 0.0) and np.any(q[1] != 0.0)
