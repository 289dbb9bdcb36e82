"""The C-ABI library loads and exports every entry point include/pagedattn.h
declares; host-side argument checks return the documented codes before any
CUDA call (so these run without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pagedattn.h")


@pytest.fixture(scope="module")
def pa():
    from paged_kv_gqa_write_gb300 import _build
    _build.build()
    import paged_kv_gqa_write_gb300 as pa
    pa.load()
    return pa


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(pa_\w+)\s*\(", src, flags=re.M)))


def _header_defines():
    vals = {}
    for m in re.finditer(r"#define\s+(PA_\w+)\s+\(?(-?\d+)\)?", open(HEADER).read()):
        vals[m.group(1)] = int(m.group(2))
    return vals


def test_every_declared_symbol_is_exported(pa):
    names = _declared()
    assert set(names) >= {"pa_kv_write", "pa_decode", "pa_prefill_chunk", "pa_combine"}
    lib = ctypes.CDLL(pa.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(pa.EXPORTED) == set(names)


def test_python_constants_match_header(pa):
    h = _header_defines()
    assert h["PA_BF16"] == pa.PA_BF16 and h["PA_F32"] == pa.PA_F32
    assert h["PA_STATUS_BAD_PAGE"] == pa.PA_STATUS_BAD_PAGE
    assert h["PA_STATUS_BAD_LENGTH"] == pa.PA_STATUS_BAD_LENGTH
    assert h["PA_STATUS_BAD_TOKENS"] == pa.PA_STATUS_BAD_TOKENS
    assert h["PA_STATUS_TIMEOUT"] == pa.PA_STATUS_TIMEOUT
    assert h["PA_MAX_CHUNKED_SEQS"] == pa.PA_MAX_CHUNKED_SEQS
    assert h["PA_SPLITS_BALANCED"] == pa.PA_SPLITS_BALANCED
    assert h["PA_BALANCED_MAX_SEQS"] == pa.PA_BALANCED_MAX_SEQS
    assert h["PA_MAX_Q_LEN"] == pa.PA_MAX_Q_LEN
    assert h["PA_MAX_PROLOGUE_HEADS"] == pa.PA_MAX_PROLOGUE_HEADS
    assert h["PA_STATUS_Q_RANGE"] == pa.PA_STATUS_Q_RANGE
    assert h["PA_PREFILL_SCHEDULE_ITEMS"] == pa.PA_PREFILL_SCHEDULE_ITEMS
    for k, v in h.items():
        if k.startswith("PA_ERR_"):
            assert getattr(pa, k) == v, k
    assert pa.pa_abi_version() == 106


def test_status_strings(pa):
    h = _header_defines()
    for k, v in h.items():
        if k.startswith("PA_ERR_"):
            s = pa.pa_status_string(v)
            assert s and s != "unknown status", k
    assert pa.pa_status_string(0) == "ok"


def _dims(pa, **kw):
    base = dict(num_seqs=2, num_q_heads=8, num_kv_heads=2, num_pages=4, max_pages_per_seq=2)
    base.update(kw)
    d = pa.make_dims(base["num_seqs"], base["num_q_heads"], base["num_kv_heads"],
                     base["num_pages"], base["max_pages_per_seq"])
    for k in ("head_dim", "page_size"):
        if k in kw:
            setattr(d, k, kw[k])
    return d


FAKE = ctypes.c_void_p(0x10000)      # never dereferenced: rejected before launch
MIS = ctypes.c_void_p(0x10008)       # 8-byte aligned only


def test_host_checks_decode(pa):
    lib, h = pa.load(), _header_defines()
    call = lambda d, q=FAKE, out=FAKE, dt=0, ns=0: lib.pa_decode(
        q, FAKE, FAKE, FAKE, FAKE, 1.0, out, dt, None, 0, ns, d, None, None)
    assert call(_dims(pa, head_dim=64)) == h["PA_ERR_HEAD_DIM"]
    assert call(_dims(pa, page_size=16)) == h["PA_ERR_PAGE_SIZE"]
    assert call(_dims(pa, num_q_heads=6, num_kv_heads=4)) == h["PA_ERR_HEADS"]
    assert call(_dims(pa, num_q_heads=34, num_kv_heads=2)) == h["PA_ERR_HEADS"]   # group 17
    assert call(_dims(pa, num_pages=0)) == h["PA_ERR_DIMS"]
    assert call(_dims(pa, num_pages=1 << 24)) == h["PA_ERR_DIMS"]
    assert call(_dims(pa), dt=7) == h["PA_ERR_OUT_DTYPE"]
    assert call(_dims(pa), ns=-2) == h["PA_ERR_SPLITS"]
    assert call(_dims(pa), q=None) == h["PA_ERR_NULL_POINTER"]
    assert call(_dims(pa), out=MIS) == h["PA_ERR_ALIGNMENT"]
    assert call(_dims(pa, num_seqs=0)) == 0                                      # nothing to do


def test_host_checks_kv_write_and_prefill(pa):
    lib, h = pa.load(), _header_defines()
    d = _dims(pa)
    assert lib.pa_kv_write(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 3, d, None, None) == h["PA_ERR_DIMS"]
    assert lib.pa_kv_write(FAKE, FAKE, None, FAKE, FAKE, FAKE, None, 2, d, None, None) == h["PA_ERR_NULL_POINTER"]
    assert lib.pa_kv_write(MIS, FAKE, FAKE, FAKE, FAKE, FAKE, None, 2, d, None, None) == h["PA_ERR_ALIGNMENT"]
    big = _dims(pa, num_seqs=h["PA_MAX_CHUNKED_SEQS"] + 1)
    assert lib.pa_kv_write(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 9, big, None, None) == h["PA_ERR_TOO_MANY_SEQS"]
    assert lib.pa_prefill_chunk(FAKE, FAKE, FAKE, FAKE, FAKE, None, 4, 1.0, FAKE, 0, d, None, None) == h["PA_ERR_NULL_POINTER"]
    assert lib.pa_prefill_chunk(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 1.0, FAKE, 3, d, None, None) == h["PA_ERR_OUT_DTYPE"]
    assert lib.pa_prefill_chunk(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, 1.0, FAKE, 0, d, None, None) == 0
    pf8 = lambda ks=FAKE, vs=FAKE, n=4, od=0: lib.pa_prefill_chunk_fp8(
        FAKE, FAKE, FAKE, ks, vs, FAKE, FAKE, FAKE, n, 1.0, FAKE, od, d, None, None)
    assert pf8(ks=None) == h["PA_ERR_NULL_POINTER"]
    assert pf8(vs=None) == h["PA_ERR_NULL_POINTER"]
    assert pf8(ks=ctypes.c_void_p(0x10002)) == h["PA_ERR_ALIGNMENT"]
    assert pf8(od=3) == h["PA_ERR_OUT_DTYPE"]
    assert pf8(n=0) == 0                                                          # nothing to do
    assert lib.pa_combine(FAKE, FAKE, 0, FAKE, 0, d, None) == h["PA_ERR_SPLITS"]
    pro = lambda eps=1e-6, base=1e6, scale=1.0, qkv=FAKE, n=2, cl=None: lib.pa_qk_norm_rope_write(
        qkv, FAKE, FAKE, eps, base, scale, 1.0, FAKE, FAKE, FAKE, FAKE, FAKE, cl, n, d, None, None)
    assert pro(eps=-1.0) == h["PA_ERR_DIMS"]
    assert pro(base=0.0) == h["PA_ERR_DIMS"]
    assert pro(scale=float("nan")) == h["PA_ERR_DIMS"]
    assert pro(n=3) == h["PA_ERR_DIMS"]                    # decode: one token per sequence
    assert pro(qkv=None) == h["PA_ERR_NULL_POINTER"]
    assert pro(qkv=MIS) == h["PA_ERR_ALIGNMENT"]
    assert pro(n=0, cl=FAKE) == 0
    pro8 = lambda ks=FAKE, vs=FAKE, n=2, eps=1e-6: lib.pa_qk_norm_rope_write_fp8(
        FAKE, FAKE, FAKE, eps, 1e6, 1.0, 1.0, FAKE, FAKE, FAKE, ks, vs, FAKE, FAKE, None, n, d,
        None, None)
    assert pro8(ks=None) == h["PA_ERR_NULL_POINTER"] and pro8(vs=None) == h["PA_ERR_NULL_POINTER"]
    assert pro8(vs=ctypes.c_void_p(0x10002)) == h["PA_ERR_ALIGNMENT"]
    assert pro8(eps=-1.0) == h["PA_ERR_DIMS"] and pro8(n=3) == h["PA_ERR_DIMS"]
    dp = lambda d=d, eps=1e-6, wq=FAKE, qkv=FAKE, od=0, ns=0, ws=None, nws=0: lib.pa_decode_prologue(
        qkv, wq, FAKE, eps, 1e6, 1.0, 1.0, FAKE, FAKE, FAKE, FAKE, 1.0, FAKE, od, ws, nws, ns, d,
        None, None)
    assert dp(eps=-1.0) == h["PA_ERR_DIMS"]
    assert dp(wq=None) == h["PA_ERR_NULL_POINTER"] and dp(qkv=None) == h["PA_ERR_NULL_POINTER"]
    assert dp(qkv=MIS) == h["PA_ERR_ALIGNMENT"] and dp(wq=MIS) == h["PA_ERR_ALIGNMENT"]
    assert dp(od=3) == h["PA_ERR_OUT_DTYPE"] and dp(ns=-2) == h["PA_ERR_SPLITS"]
    assert dp(d=_dims(pa, num_q_heads=34, num_kv_heads=2)) == h["PA_ERR_HEADS"]   # G = 17
    assert dp(d=_dims(pa, num_seqs=0)) == 0
    wide = _dims(pa, num_q_heads=352, num_kv_heads=32)  # G = 11, 416 heads in a row
    assert lib.pa_qk_norm_rope_write(FAKE, FAKE, FAKE, 1e-6, 1e6, 1.0, 1.0, FAKE, FAKE, FAKE, FAKE,
                                     FAKE, None, 2, wide, None, None) == h["PA_ERR_HEADS"]
    tk = lambda rows=2, vocab=100, k=8, stride=100, ptr=FAKE: lib.pa_topk(
        ptr, stride, rows, vocab, k, FAKE, FAKE, FAKE, 1 << 20, None)
    assert tk(k=0) == h["PA_ERR_DIMS"] and tk(k=33) == h["PA_ERR_DIMS"]
    assert tk(vocab=4, k=8) == h["PA_ERR_DIMS"] and tk(stride=50) == h["PA_ERR_DIMS"]
    assert tk(ptr=None) == h["PA_ERR_NULL_POINTER"]
    assert tk(ptr=ctypes.c_void_p(0x10002)) == h["PA_ERR_ALIGNMENT"]
    assert tk(rows=0) == 0
    assert h["PA_TOPK_MAX_K"] == pa.PA_TOPK_MAX_K
    assert lib.pa_combine(FAKE, FAKE, 2, MIS, 0, d, None) == h["PA_ERR_ALIGNMENT"]


def test_workspace_size_invalid_dims(pa):
    assert pa.load().pa_decode_workspace_size(_dims(pa, head_dim=64), 2) == ctypes.c_size_t(-1).value


def test_decode_multi_rejects_q_len_on_the_host(pa):
    """q_len outside 1..PA_MAX_Q_LEN is refused before any device work."""
    lib = ctypes.CDLL(pa.LIB_PATH)
    lib.pa_decode_multi.restype = ctypes.c_int
    lib.pa_decode_multi_workspace_size.restype = ctypes.c_size_t
    d = pa.make_dims(4, 40, 8, 64, 16)
    for bad in (0, -1, pa.PA_MAX_Q_LEN + 1):
        rc = lib.pa_decode_multi(None, None, None, None, None, ctypes.c_int32(bad),
                                 ctypes.c_float(0.1), None, ctypes.c_int32(pa.PA_BF16), None,
                                 ctypes.c_size_t(0), ctypes.c_int32(1), d, None, None)
        assert rc == pa.PA_ERR_DIMS, (bad, rc)
        n = lib.pa_decode_multi_workspace_size(d, ctypes.c_int32(bad), ctypes.c_int32(1))
        assert n == ctypes.c_size_t(-1).value


def test_host_checks_wait_selftest_and_noalloc(pa):
    """pa_wait_selftest refuses a limit out of range or a NULL status, and
    pa_decode_noalloc shares pa_decode's checks (including the 32-bit row
    bound), all before any launch."""
    lib, h = pa.load(), _header_defines()
    assert lib.pa_wait_selftest(0, FAKE, None) == h["PA_ERR_DIMS"]
    assert lib.pa_wait_selftest(5000001, FAKE, None) == h["PA_ERR_DIMS"]
    assert lib.pa_wait_selftest(1000, None, None) == h["PA_ERR_NULL_POINTER"]
    na = lambda d, q=FAKE, out=FAKE, dt=0, ns=0: lib.pa_decode_noalloc(
        q, FAKE, FAKE, FAKE, FAKE, 1.0, out, dt, ns, d, None, None)
    assert na(_dims(pa, head_dim=64)) == h["PA_ERR_HEAD_DIM"]
    assert na(_dims(pa), dt=7) == h["PA_ERR_OUT_DTYPE"]
    assert na(_dims(pa), ns=-2) == h["PA_ERR_SPLITS"]
    assert na(_dims(pa), q=None) == h["PA_ERR_NULL_POINTER"]
    assert na(_dims(pa), out=MIS) == h["PA_ERR_ALIGNMENT"]
    assert na(_dims(pa, num_seqs=0)) == 0
    # B * Hq rows beyond int32: refused like pa_decode (no scratch is needed
    # with one split, so the size check alone would not catch it)
    huge = _dims(pa, num_seqs=40_000_000, num_q_heads=128, num_kv_heads=8)
    assert na(huge, ns=1) == h["PA_ERR_DIMS"]
    assert lib.pa_decode(FAKE, FAKE, FAKE, FAKE, FAKE, 1.0, FAKE, 0, None, 0, 1, huge, None,
                         None) == h["PA_ERR_DIMS"]
