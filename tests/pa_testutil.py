"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and
the FP64 oracle on the same bits, and compare."""
import numpy as np
import torch

import oracle

# Attention output tolerance vs the FP64 oracle with FP32 output (BF16 inputs,
# FP32 accumulation).
ATOL = 5e-3
# P5-style cross-check thresholds (rel-L2 over a whole output).
REL_L2 = 8e-3


# (test, what, max|err|, bound) of every comparison made through the helpers
# below; tests/conftest.py prints them at the end of the run and, when
# PA_MAXERR_LOG names a file, writes them there as JSON.
ERRORS = []


def _record(what, mx, bound):
    import os
    test = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]
    ERRORS.append((test, what, float(mx), float(bound)))


def dev_status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def oracle_decode(case, rows=None, threads=None):
    return oracle.attention(case.q, case.k_cache, case.v_cache, case.block_table,
                            case.context_lens, None, case.scale, case.Hq, case.Hkv,
                            case.num_pages, case.max_pages_per_seq, rows=rows,
                            num_threads=threads)


def oracle_prefill(case, rows=None, threads=None):
    return oracle.attention(case.q, case.k_cache, case.v_cache, case.block_table,
                            case.context_lens, case.chunk_lens, case.scale, case.Hq, case.Hkv,
                            case.num_pages, case.max_pages_per_seq, rows=rows,
                            num_threads=threads)


def assert_close(gpu, ref, atol=ATOL, what=""):
    g = gpu.detach().float().cpu().double().numpy().reshape(ref.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    err = np.abs(g - ref)
    mx = float(err.max()) if err.size else 0.0
    _record(what, mx, atol)
    assert mx <= atol, f"{what}: max|err| {mx:.3e} > {atol:.1e} at {np.unravel_index(err.argmax(), err.shape)}"
    denom = np.linalg.norm(ref)
    if denom > 0:
        rel = np.linalg.norm(g - ref) / denom
        assert rel < REL_L2, f"{what}: rel-L2 {rel:.3e}"
    return mx


def assert_close_bf16(gpu, ref, what=""):
    """BF16 output: the FP32 result rounded to bf16 -> within the FP32 tolerance
    plus one half bf16 ulp of the value."""
    g = gpu.detach().float().cpu().double().numpy().reshape(ref.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    bound = ATOL + np.abs(ref) * 2.0 ** -8
    err = np.abs(g - ref)
    # recorded: the worst error as a fraction of its element's bound
    _record(what + " (bf16 out, err / bound)", float((err / bound).max()) if err.size else 0.0, 1.0)
    bad = err > bound
    assert not bad.any(), f"{what}: {bad.sum()} elements beyond bf16 bound"


def cache_bits(t):
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def sample_rows(T, Hq, n, seed, extra=()):
    rng = np.random.default_rng(seed)
    ids = set(int(x) for x in rng.choice(T * Hq, size=min(n, T * Hq), replace=False))
    ids.update([0, T * Hq - 1, *extra])
    return np.array(sorted(i for i in ids if 0 <= i < T * Hq), dtype=np.int64)
