"""Pins for the oracle's exact top-k (pypto-serving PR #77, "Exactness Design":
an exact Top-32 of full-vocabulary logits, checked against torch.topk; its two
adversarial fixtures).  Checked against brute force on small rows, against the
selection invariants, against the page's fixtures, and on ties and infinities."""
import numpy as np
import pytest

import oracle

VOCAB = 151936  # Qwen3-14B real vocabulary (the page's row width)


def _brute(row, k):
    """k rounds of 'take the largest remaining value, smallest index on ties'."""
    row = np.array(row, dtype=np.float64)
    taken = np.zeros(row.shape[0], dtype=bool)
    vals, idx = [], []
    for _ in range(k):
        best = -1
        for i in range(row.shape[0]):
            if taken[i]:
                continue
            if best < 0:
                best = i
                continue
            a, b = row[i], row[best]
            if np.isnan(a) and not np.isnan(b):
                best = i
            elif not np.isnan(a) and not np.isnan(b) and a > b:
                best = i
        taken[best] = True
        vals.append(row[best]); idx.append(best)
    return np.array(vals, dtype=np.float32), np.array(idx, dtype=np.int32)


def _check_invariants(x, vals, idx, k):
    rows, vocab = x.shape
    for r in range(rows):
        assert len(set(idx[r].tolist())) == k
        assert np.array_equal(vals[r], x[r, idx[r]])
        rest = np.setdiff1d(np.arange(vocab), idx[r])
        if rest.size:
            assert np.nanmin(vals[r]) >= np.nanmax(x[r, rest]) or np.isnan(vals[r]).all()
        # descending, ties by index
        for j in range(k - 1):
            a, b = vals[r, j], vals[r, j + 1]
            assert a > b or (a == b and idx[r, j] < idx[r, j + 1]) or np.isnan(a)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_small_rows_match_brute_force(seed):
    rng = np.random.default_rng(seed)
    x = rng.integers(-8, 8, size=(4, 97)).astype(np.float32)  # many ties
    for k in (1, 5, 32):
        vals, idx = oracle.topk(x, k)
        for r in range(x.shape[0]):
            bv, bi = _brute(x[r], k)
            assert np.array_equal(vals[r], bv) and np.array_equal(idx[r], bi)


def test_full_vocabulary_invariants_and_numpy_agreement():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((2, VOCAB)).astype(np.float32)
    vals, idx = oracle.topk(x, 32)
    _check_invariants(x, vals, idx, 32)
    # continuous data has no ties: the result equals a stable argsort of -x
    ref = np.argsort(-x, axis=1, kind="stable")[:, :32]
    assert np.array_equal(idx, ref)


def test_page_fixture_all_winners_in_one_512_region():
    rng = np.random.default_rng(4)
    x = rng.uniform(-1.0, 0.0, size=(1, VOCAB)).astype(np.float32)
    base = 512 * 137
    x[0, base:base + 32] = np.linspace(10.0, 5.0, 32, dtype=np.float32)
    vals, idx = oracle.topk(x, 32)
    assert np.array_equal(idx[0], np.arange(base, base + 32, dtype=np.int32))


def test_page_fixture_one_winner_per_chunk():
    rng = np.random.default_rng(5)
    x = rng.uniform(-1.0, 0.0, size=(1, VOCAB)).astype(np.float32)
    chunks = rng.choice(VOCAB // 512, size=32, replace=False)
    pos = chunks * 512 + rng.integers(0, 512, size=32)
    x[0, pos] = np.arange(100, 132, dtype=np.float32)[::-1]
    vals, idx = oracle.topk(x, 32)
    assert np.array_equal(idx[0], pos.astype(np.int32))
    assert np.array_equal(vals[0], np.arange(100, 132, dtype=np.float32)[::-1])


def test_ties_and_infinities():
    x = np.zeros((1, 1000), dtype=np.float32)
    vals, idx = oracle.topk(x, 32)
    assert np.array_equal(idx[0], np.arange(32))          # all equal: smallest indices
    x[0, 500] = np.inf
    x[0, 700] = np.nan
    x[0, 10] = -np.inf
    vals, idx = oracle.topk(x, 3)
    assert idx[0].tolist() == [700, 500, 0]
    assert np.isnan(vals[0, 0]) and vals[0, 1] == np.inf and vals[0, 2] == 0.0
