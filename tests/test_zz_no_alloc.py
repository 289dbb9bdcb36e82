"""pa_decode_noalloc: the decode entry point for callers that cannot allocate
device memory (for example a plugin whose host framework owns every buffer,
or a latency-critical path that must not call cudaMalloc).  It must give the
same results as pa_decode with a caller workspace, call after call, even
though every call reuses the library's one scratch array.

Collected last on purpose, so a run that stops at the first failure has run
every other test before this one."""
import ctypes

import pytest
import torch

import workloads as W
from pa_testutil import ATOL, assert_close, dev_status, oracle_decode

pytestmark = pytest.mark.gpu


def _noalloc_via_abi(lib, c, out, splits):
    """Call the C entry point directly with raw device pointers."""
    st = dev_status()
    d = lib.make_dims(c.B, c.Hq, c.Hkv, c.num_pages, c.max_pages_per_seq)
    rc = lib.load().pa_decode_noalloc(
        ctypes.c_void_p(c.q.data_ptr()), ctypes.c_void_p(c.k_cache.data_ptr()),
        ctypes.c_void_p(c.v_cache.data_ptr()), ctypes.c_void_p(c.block_table.data_ptr()),
        ctypes.c_void_p(c.context_lens.data_ptr()), ctypes.c_float(c.scale),
        ctypes.c_void_p(out.data_ptr()), lib.PA_F32, int(splits), d,
        ctypes.c_void_p(st.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return rc, int(st.item())


def _reference(lib, c, splits):
    out = lib.pa_decode(c.q, c.k_cache, c.v_cache, c.block_table, c.context_lens, c.scale,
                        out_dtype=torch.float32, num_splits=splits)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("splits", [0, 4])
def test_two_calls_in_a_row_match_pa_decode(cuda_lib, splits):
    # two different inputs back to back: the second call must not see the
    # first call's leftovers in the shared scratch array
    cases = [W.qwen3_14b_decode_b16().to("cuda"),
             W.custom_case(901, [4096, 1, 0, 700, 129], Hq=40, Hkv=8,
                           max_pages_per_seq=32).to("cuda")]
    for c in cases:
        ref = _reference(cuda_lib, c, splits)
        out = torch.full_like(ref, float("nan"))
        rc, st = _noalloc_via_abi(cuda_lib, c, out, splits)
        assert rc == 0, cuda_lib.pa_status_string(rc)
        assert st == 0
        assert_close(out, ref.double().cpu().numpy(), atol=ATOL, what=f"noalloc s={splits}")


def test_rejects_sizes_beyond_the_scratch_array(cuda_lib):
    # 2048 sequences x 64 heads x 32 splits of partials is far beyond 16 MiB;
    # rejected on the host before any launch
    c = W.tiny_decode().to("cuda")
    big = cuda_lib.make_dims(2048, 64, 8, 4096, 32)
    fake = ctypes.c_void_p(c.q.data_ptr())
    rc = cuda_lib.load().pa_decode_noalloc(fake, fake, fake, fake, fake, ctypes.c_float(1.0),
                                           fake, cuda_lib.PA_F32, 32, big, None, None)
    assert rc == -13
    assert "PA_NOALLOC_SCRATCH_BYTES" in cuda_lib.pa_status_string(rc)


def test_python_wrapper_balanced_matches_the_oracle(cuda_lib):
    # the binding's pa_decode_noalloc with an explicit page-balanced schedule,
    # twice in a row on different inputs, each checked against the FP64 oracle
    cases = [W.custom_case(902, [4096, 3000, 17, 1, 2500, 129, 0, 640], Hq=40, Hkv=8,
                           max_pages_per_seq=32),
             W.custom_case(903, [100, 4096, 4096, 300], Hq=64, Hkv=8, max_pages_per_seq=32)]
    for case in cases:
        c = case.to("cuda")
        out = torch.full((case.B, case.Hq, 128), float("nan"), dtype=torch.float32,
                         device="cuda")
        st = dev_status()
        cuda_lib.pa_decode_noalloc(c.q, c.k_cache, c.v_cache, c.block_table, c.context_lens,
                                   c.scale, out=out, num_splits=cuda_lib.PA_SPLITS_BALANCED,
                                   status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert_close(out, oracle_decode(case), atol=ATOL, what="noalloc balanced vs oracle")


def test_python_wrapper_rejects_other_out_dtypes(cuda_lib):
    c = W.tiny_decode().to("cuda")
    out = torch.empty(c.B, c.Hq, 128, dtype=torch.float16, device="cuda")
    with pytest.raises(TypeError):
        cuda_lib.pa_decode_noalloc(c.q, c.k_cache, c.v_cache, c.block_table, c.context_lens,
                                   c.scale, out=out)
