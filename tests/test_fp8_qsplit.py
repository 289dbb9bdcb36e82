"""The query split of the FP8-cache kernels, checked on the CPU over every
finite bf16 value.

pa_decode_fp8 and pa_prefill_chunk_fp8 run q . K on the e4m3 K codes, so the
query side is e4m3 too: each element q (bf16) of a row whose largest
magnitude is M is scaled by x = 2^(134 - e(M)) (e(M) the biased exponent of
M's bf16 bits, x capped at 2^126) and split into hi = e4m3(x q) and
lo = e4m3(x q - hi), both rounded to nearest.  The kernels' headers state that
hi + lo = x q exactly for every element with |x q| >= 2^-2 (i.e. within 2^10
of the largest) and that the others are off by at most 2^-10 in the scaled
unit.  This test restates the split with torch's float8_e4m3fn conversion
(round to nearest even) and checks both statements for all 65280 finite bf16
values against several maxima, including the largest and a subnormal one.
"""
import pytest
import torch


def _finite_bf16():
    bits = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16)
    v = bits.view(torch.bfloat16).float()
    return v[torch.isfinite(v)]


def _scale(amax):
    """x for a row whose largest |q| is amax: the largest goes to [128, 256)."""
    be = int((torch.tensor(amax, dtype=torch.bfloat16).view(torch.int16).int() & 0x7FFF) >> 7)
    return 2.0 ** min(134 - be, 126)


def _split(q, x):
    a = (q.double() * x).float()  # exact: a power of two, no overflow below 256
    hi = a.to(torch.float8_e4m3fn).float()
    lo = (a - hi).to(torch.float8_e4m3fn).float()  # a - hi is exact in float
    return a.double(), hi.double(), lo.double()


@pytest.mark.parametrize("amax", [1.0, 3.7, 0.0884, 448.0, 1.0e-30, 2.5e38, 1.0e-39])
def test_split_is_exact_near_the_row_maximum(amax):
    v = _finite_bf16()
    q = v[v.abs() <= torch.tensor(amax, dtype=torch.bfloat16).float()]
    x = _scale(amax)
    a, hi, lo = _split(q, x)
    assert a.abs().max() < 256.0  # no element reaches the e4m3 saturation range
    assert torch.isfinite(hi).all() and torch.isfinite(lo).all()
    err = (hi + lo - a).abs()
    near = a.abs() >= 0.25
    if x < 2.0 ** 126:  # (a subnormal maximum caps x: then no element is near)
        assert bool(near.any())
    if bool(near.any()):
        assert float(err[near].max()) == 0.0
    assert float(err.max()) <= 2.0 ** -10


def test_scaled_maximum_lies_in_128_256():
    v = _finite_bf16()
    pos = v[(v > 0) & (v >= 2.0 ** -119)]  # x below its 2^126 cap
    for m in pos[:: 97]:
        x = _scale(float(m))
        assert 128.0 <= float(m) * x < 256.0


def test_power_of_two_rescaling_gives_the_same_codes():
    """q and q times 2^15 split into the same e4m3 codes (the scale absorbs the
    factor): the basis of the GPU tests that compare the two calls bit for bit."""
    g = torch.Generator().manual_seed(5)
    q = torch.randn(4096, generator=g).to(torch.bfloat16).float()
    big = (q * 2.0 ** 15).to(torch.bfloat16).float()
    assert torch.equal(big, q * 2.0 ** 15)
    m, mb = float(q.abs().max()), float(big.abs().max())
    _, hi, lo = _split(q, _scale(m))
    _, hib, lob = _split(big, _scale(mb))
    assert torch.equal(hi, hib) and torch.equal(lo, lob)
    assert _scale(m) == _scale(mb) * 2.0 ** 15
