"""pa_topk (exact top-k of logit rows) on the GPU against the oracle, bit for
bit: the indices and the values (the logits as given) of every row."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu
VOCAB = 151936          # Qwen3-14B real vocabulary
PADDED = 152064         # its padded row (the page compares logits[:, :REAL_VOCAB])


def _same(a, b):
    a, b = np.asarray(a), np.asarray(b)
    return np.array_equal(np.isnan(a), np.isnan(b)) and np.array_equal(a[~np.isnan(a)], b[~np.isnan(b)])


def _check(pa, x, k, stride=None):
    rows, vocab = x.shape
    if stride is None:
        xt = torch.from_numpy(x).cuda()
    else:
        buf = torch.full((rows, stride), -7.0, dtype=torch.float32)
        buf[:, :vocab] = torch.from_numpy(x)
        xt = buf.cuda()[:, :vocab]
    vals, idx = pa.pa_topk(xt, k)
    torch.cuda.synchronize()
    rv, ri = oracle.topk(x, k)
    gi, gv = idx.cpu().numpy(), vals.cpu().numpy()
    assert np.array_equal(gi, ri), f"indices differ in {np.sum(np.any(gi != ri, axis=1))} rows"
    assert _same(gv, rv)


@pytest.mark.parametrize("k", [32, 1, 7])
def test_full_vocabulary_batch16(cuda_lib, k):
    x = np.random.default_rng(700 + k).standard_normal((16, VOCAB)).astype(np.float32)
    _check(cuda_lib, x, k, stride=PADDED)


def test_page_fixture_all_winners_in_one_512_region(cuda_lib):
    rng = np.random.default_rng(701)
    x = rng.uniform(-1.0, 0.0, size=(4, VOCAB)).astype(np.float32)
    for r in range(4):
        base = 512 * int(rng.integers(0, VOCAB // 512))
        x[r, base:base + 32] = np.linspace(10.0, 5.0, 32, dtype=np.float32)
    _check(cuda_lib, x, 32)


def test_page_fixture_one_winner_per_chunk(cuda_lib):
    rng = np.random.default_rng(702)
    x = rng.uniform(-1.0, 0.0, size=(4, VOCAB)).astype(np.float32)
    for r in range(4):
        chunks = rng.choice(VOCAB // 512, size=32, replace=False)
        x[r, chunks * 512 + rng.integers(0, 512, size=32)] = rng.uniform(50, 60, 32)
    _check(cuda_lib, x, 32)


def test_heavy_ties_break_by_index(cuda_lib):
    rng = np.random.default_rng(703)
    x = rng.integers(-8, 9, size=(8, VOCAB)).astype(np.float32)
    _check(cuda_lib, x, 32)
    _check(cuda_lib, np.zeros((2, 50000), dtype=np.float32), 32)


def test_nan_infinities_and_signed_zero(cuda_lib):
    x = np.zeros((3, 70000), dtype=np.float32)
    x[0, 123] = np.nan
    x[0, 40000] = np.inf
    x[0, 5] = -np.inf
    x[1, :] = -np.inf
    x[1, 69999] = -0.0
    x[1, 3] = 0.0
    x[2, ::2] = -0.0
    _check(cuda_lib, x, 32)


@pytest.mark.parametrize("vocab,k", [(32, 32), (40, 32), (1000, 5), (5000, 32), (16385, 32)])
def test_small_and_ragged_vocabularies(cuda_lib, vocab, k):
    x = np.random.default_rng(704 + vocab).standard_normal((5, vocab)).astype(np.float32)
    _check(cuda_lib, x, k)


def test_many_rows(cuda_lib):
    x = np.random.default_rng(705).standard_normal((300, 4096)).astype(np.float32)
    _check(cuda_lib, x, 32)
