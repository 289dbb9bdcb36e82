"""FP64 CPU oracle for paged-KV GQA attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or runs it; the two share no code.

The arithmetic lives in ``pa_oracle.c`` (plain C, double precision); this
module only marshals numpy arrays of bfloat16 bit patterns (uint16) into it.
See that file's header for the sources and readings each function follows.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        i32p = np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")
        u16p = np.ctypeslib.ndpointer(np.uint16, flags="C_CONTIGUOUS")
        f64p = np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")
        c_int, c_i64, c_dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.oracle_kv_write.restype = c_int
        lib.oracle_kv_write.argtypes = [u16p, u16p, u16p, u16p, i32p, i32p, ctypes.c_void_p,
                                        c_i64, c_int, c_int, c_int, c_int, c_int, c_int]
        lib.oracle_attention.restype = c_int
        lib.oracle_attention.argtypes = [u16p, u16p, u16p, i32p, i32p, ctypes.c_void_p,
                                         c_int, c_int, c_int, c_int, c_int, c_int, c_int,
                                         c_dbl, ctypes.c_void_p, c_i64, f64p, c_int]
        lib.oracle_dense_attention.restype = None
        lib.oracle_dense_attention.argtypes = [f64p, f64p, f64p, c_i64, c_int, c_dbl, f64p,
                                               ctypes.POINTER(c_dbl), f64p]
        lib.oracle_combine.restype = None
        lib.oracle_combine.argtypes = [f64p, f64p, c_i64, c_int, c_int, f64p]
        f32p = np.ctypeslib.ndpointer(np.float32, flags="C_CONTIGUOUS")
        lib.oracle_qk_norm_rope_write.restype = c_int
        lib.oracle_qk_norm_rope_write.argtypes = [u16p, f32p, f32p, c_dbl, c_dbl, c_dbl, c_dbl,
                                                  f64p, u16p, u16p, i32p, i32p, ctypes.c_void_p,
                                                  c_i64, c_int, c_int, c_int, c_int, c_int,
                                                  c_int, c_int]
        lib.oracle_rope_neox.restype = None
        lib.oracle_rope_neox.argtypes = [f64p, c_int, c_dbl, c_dbl, c_dbl]
        lib.oracle_topk.restype = None
        lib.oracle_topk.argtypes = [f32p, c_i64, c_int, c_int, c_int, f32p, i32p]
        u8p = np.ctypeslib.ndpointer(np.uint8, flags="C_CONTIGUOUS")
        lib.oracle_e4m3_encode_array.restype = None
        lib.oracle_e4m3_encode_array.argtypes = [f32p, c_i64, u8p]
        lib.oracle_e4m3_decode_array.restype = None
        lib.oracle_e4m3_decode_array.argtypes = [u8p, c_i64, f64p]
        lib.oracle_kv_write_fp8.restype = c_int
        lib.oracle_kv_write_fp8.argtypes = [u16p, u16p, u8p, u8p, f32p, f32p, i32p, i32p,
                                            ctypes.c_void_p, c_i64, c_int, c_int, c_int, c_int,
                                            c_int, c_int]
        lib.oracle_attention_fp8.restype = c_int
        lib.oracle_attention_fp8.argtypes = [u16p, u8p, u8p, f32p, f32p, i32p, i32p,
                                             ctypes.c_void_p, c_int, c_int, c_int, c_int, c_int,
                                             c_int, c_int, c_dbl, ctypes.c_void_p, c_i64, f64p,
                                             c_int]
        lib.oracle_max_threads.restype = c_int
        lib.oracle_max_threads.argtypes = []
        _lib = lib
    return _lib


def _u16(a):
    """bf16 data as a C-contiguous uint16 numpy view (accepts torch or numpy)."""
    if hasattr(a, "detach"):  # torch tensor
        import torch
        a = a.detach().cpu().contiguous()
        if a.dtype == torch.bfloat16:
            a = a.view(torch.int16)
        return np.ascontiguousarray(a.numpy().view(np.uint16))
    a = np.ascontiguousarray(a)
    assert a.dtype.itemsize == 2, a.dtype
    return a.view(np.uint16)


def _i32(a):
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.int32)


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def kv_write(k_new, v_new, k_cache, v_cache, block_table, context_lens, chunk_lens,
             num_pages, max_pages_per_seq, page_size=128):
    """Returns (k_cache', v_cache', skipped) with the new tokens' rows copied into
    their slots (uint16 arrays); the inputs are not modified."""
    kc = _u16(k_cache).copy()
    vc = _u16(v_cache).copy()
    kn, vn = _u16(k_new), _u16(v_new)
    row = kc.shape[-2] * kc.shape[-1]
    T = kn.size // row
    ctx = _i32(context_lens)
    B = ctx.shape[0]
    hkv, d = kc.shape[-2], kc.shape[-1]
    cl = None if chunk_lens is None else _i32(chunk_lens)
    skipped = _load().oracle_kv_write(
        kn, vn, kc, vc, _i32(block_table).reshape(-1), ctx,
        None if cl is None else cl.ctypes.data_as(ctypes.c_void_p),
        T, B, hkv, d, page_size, num_pages, max_pages_per_seq)
    return kc, vc, skipped


def attention(q, k_cache, v_cache, block_table, context_lens, chunk_lens, scale,
              num_q_heads, num_kv_heads, num_pages, max_pages_per_seq, rows=None,
              num_threads=None, page_size=128, head_dim=128):
    """Paged attention in float64.  q is [T, Hq, D] (decode: T = B, chunk_lens=None).
    Returns [T, Hq, D] float64, or [len(rows), D] for the (token*Hq + head) ids in rows."""
    qq = _u16(q).reshape(-1)
    kc, vc = _u16(k_cache).reshape(-1), _u16(v_cache).reshape(-1)
    ctx = _i32(context_lens)
    B = ctx.shape[0]
    cl = None if chunk_lens is None else _i32(chunk_lens)
    T = B if cl is None else int(np.maximum(cl, 0).sum())
    if rows is None:
        nrows, rp, out_shape = T * num_q_heads, None, (T, num_q_heads, head_dim)
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        nrows, rp, out_shape = rows.shape[0], rows.ctypes.data_as(ctypes.c_void_p), (rows.shape[0], head_dim)
    out = np.zeros((max(nrows, 1), head_dim), dtype=np.float64)
    nt = num_threads if num_threads is not None else max_threads()
    rc = _load().oracle_attention(
        qq, kc, vc, _i32(block_table).reshape(-1), ctx,
        None if cl is None else cl.ctypes.data_as(ctypes.c_void_p),
        B, num_q_heads, num_kv_heads, head_dim, page_size, num_pages, max_pages_per_seq,
        float(scale), rp, nrows, out, int(nt))
    if rc != 0:
        raise ValueError("oracle_attention: bad row index")
    return out[:nrows].reshape(out_shape)


def _u8(a):
    """FP8 cache data as a C-contiguous uint8 numpy view (torch uint8/float8 or numpy)."""
    if hasattr(a, "detach"):
        import torch
        a = a.detach().cpu().contiguous()
        if a.dtype != torch.uint8:
            a = a.view(torch.uint8)
        return np.ascontiguousarray(a.numpy())
    a = np.ascontiguousarray(a)
    assert a.dtype.itemsize == 1, a.dtype
    return a.view(np.uint8)


def _f32(a):
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.float32)


def e4m3_encode(x):
    """Nearest e4m3 codes (uint8) of float32 values: ties to even, saturating at
    +-448, NaN to a NaN code."""
    x = _f32(x)
    out = np.empty(x.shape, dtype=np.uint8)
    _load().oracle_e4m3_encode_array(x.reshape(-1), x.size, out.reshape(-1))
    return out


def e4m3_decode(codes):
    """Exact float64 values of e4m3 codes."""
    c = _u8(codes)
    out = np.empty(c.shape, dtype=np.float64)
    _load().oracle_e4m3_decode_array(c.reshape(-1), c.size, out.reshape(-1))
    return out


def kv_write_fp8(k_new, v_new, k_cache, v_cache, k_scale, v_scale, block_table, context_lens,
                 chunk_lens, num_pages, max_pages_per_seq, page_size=128):
    """FP8 KV write: returns (k_cache', v_cache', skipped), uint8 e4m3 caches with
    the new tokens' rows quantized (bf16 value / per-head FP32 scale) into their
    slots; the inputs are not modified."""
    kc = _u8(k_cache).copy()
    vc = _u8(v_cache).copy()
    kn, vn = _u16(k_new), _u16(v_new)
    hkv, d = kc.shape[-2], kc.shape[-1]
    T = kn.size // (hkv * d)
    ctx = _i32(context_lens)
    cl = None if chunk_lens is None else _i32(chunk_lens)
    skipped = _load().oracle_kv_write_fp8(
        kn, vn, kc, vc, _f32(k_scale), _f32(v_scale), _i32(block_table).reshape(-1), ctx,
        None if cl is None else cl.ctypes.data_as(ctypes.c_void_p),
        T, ctx.shape[0], hkv, d, page_size, num_pages, max_pages_per_seq)
    return kc, vc, skipped


def attention_fp8(q, k_cache, v_cache, k_scale, v_scale, block_table, context_lens, chunk_lens,
                  scale, num_q_heads, num_kv_heads, num_pages, max_pages_per_seq, rows=None,
                  num_threads=None, page_size=128, head_dim=128):
    """Paged attention in float64 over an FP8 cache (uint8 e4m3 codes, per-KV-head
    FP32 scales).  Same shapes and row selection as attention()."""
    qq = _u16(q).reshape(-1)
    kc, vc = _u8(k_cache).reshape(-1), _u8(v_cache).reshape(-1)
    ctx = _i32(context_lens)
    B = ctx.shape[0]
    cl = None if chunk_lens is None else _i32(chunk_lens)
    T = B if cl is None else int(np.maximum(cl, 0).sum())
    if rows is None:
        nrows, rp, out_shape = T * num_q_heads, None, (T, num_q_heads, head_dim)
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        nrows, rp, out_shape = rows.shape[0], rows.ctypes.data_as(ctypes.c_void_p), (rows.shape[0], head_dim)
    out = np.zeros((max(nrows, 1), head_dim), dtype=np.float64)
    nt = num_threads if num_threads is not None else max_threads()
    rc = _load().oracle_attention_fp8(
        qq, kc, vc, _f32(k_scale), _f32(v_scale), _i32(block_table).reshape(-1), ctx,
        None if cl is None else cl.ctypes.data_as(ctypes.c_void_p),
        B, num_q_heads, num_kv_heads, head_dim, page_size, num_pages, max_pages_per_seq,
        float(scale), rp, nrows, out, int(nt))
    if rc != 0:
        raise ValueError("oracle_attention_fp8: bad row index")
    return out[:nrows].reshape(out_shape)


def dense_attention(q, K, V, scale):
    """One query q [D] over dense keys K, V [n, D] (float64). Returns (out [D], lse)."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    K = np.ascontiguousarray(K, dtype=np.float64).reshape(-1, q.shape[0])
    V = np.ascontiguousarray(V, dtype=np.float64).reshape(-1, q.shape[0])
    out = np.zeros(q.shape[0], dtype=np.float64)
    lse = ctypes.c_double(0.0)
    x = np.zeros(max(K.shape[0], 1), dtype=np.float64)
    _load().oracle_dense_attention(q, K, V, K.shape[0], q.shape[0], float(scale), out,
                                   ctypes.byref(lse), x)
    return out, lse.value


def combine(part_o, part_lse):
    """part_o [R, S, D], part_lse [R, S] (float64) -> [R, D] LSE-weighted merge."""
    po = np.ascontiguousarray(part_o, dtype=np.float64)
    pl = np.ascontiguousarray(part_lse, dtype=np.float64)
    R, S, D = po.shape
    out = np.zeros((max(R, 1), D), dtype=np.float64)
    _load().oracle_combine(po, pl, R, S, D, out)
    return out[:R]


def rope_neox(x, pos, base, scale=1.0):
    """NeoX rotary embedding of one head vector x [D] (float64) at position pos."""
    y = np.array(x, dtype=np.float64, copy=True)
    _load().oracle_rope_neox(y, y.shape[0], float(pos), float(base), float(scale))
    return y


def qk_norm_rope_write(qkv, q_norm_w, k_norm_w, k_cache, v_cache, block_table,
                       context_lens, chunk_lens, num_q_heads, num_kv_heads, num_pages,
                       max_pages_per_seq, eps=1e-6, rope_base=1e6, rope_scale=1.0,
                       q_scale=1.0, page_size=128, head_dim=128):
    """The prologue: per-head RMSNorm of Q and K, NeoX RoPE at each token's
    position, Q times q_scale; K (bf16-rounded) and V written to their slots.
    qkv is [T, (Hq + 2 Hkv) * D] bf16.  Returns (q_out [T, Hq, D] float64,
    k_cache', v_cache', skipped); the caches passed in are not modified."""
    x = _u16(qkv).reshape(-1)
    T = x.size // ((num_q_heads + 2 * num_kv_heads) * head_dim)
    kc = _u16(k_cache).copy()
    vc = _u16(v_cache).copy()
    ctx = _i32(context_lens)
    cl = None if chunk_lens is None else _i32(chunk_lens)
    q_out = np.zeros((max(T, 1), num_q_heads, head_dim), dtype=np.float64)
    wq = np.ascontiguousarray(q_norm_w, dtype=np.float32)
    wk = np.ascontiguousarray(k_norm_w, dtype=np.float32)
    skipped = _load().oracle_qk_norm_rope_write(
        x, wq, wk, float(eps), float(rope_base), float(rope_scale), float(q_scale), q_out,
        kc.reshape(-1), vc.reshape(-1), _i32(block_table).reshape(-1), ctx,
        None if cl is None else cl.ctypes.data_as(ctypes.c_void_p),
        T, ctx.shape[0], num_q_heads, num_kv_heads, head_dim, page_size, num_pages,
        max_pages_per_seq)
    return q_out[:T], kc, vc, skipped


def qk_norm_rope_write_fp8(qkv, q_norm_w, k_norm_w, k_cache, v_cache, k_scale, v_scale,
                           block_table, context_lens, chunk_lens, num_q_heads, num_kv_heads,
                           num_pages, max_pages_per_seq, eps=1e-6, rope_base=1e6,
                           rope_scale=1.0, q_scale=1.0, page_size=128, head_dim=128):
    """The prologue over an FP8 (e4m3) cache: the rows qk_norm_rope_write stores
    (K normed, rotated and rounded to bf16; V as given), each quantized as
    kv_write_fp8 quantizes a bf16 row -- element d of KV head h becomes the
    e4m3 code of (float)x / scale[h], an FP32 quotient.  The "fp8_e4m3" KV
    cache of the "Qwen4-Exp QSA" blog (DGX Spark note) written by the prologue
    of "Qwen 3" (TensorSharp) section 3 / "Qwen3-14B" decode_fwd.  k_cache and
    v_cache are uint8 [num_pages, page_size, Hkv, D]; returns (q_out float64,
    k_cache', v_cache', skipped), the caches passed in unmodified.

    A slot is written when the bf16 prologue, run on two scratch caches of
    opposite fill (all-zero and all-ones bits), leaves the same row in both:
    a stored row does not depend on what the slot held before."""
    kc8 = _u8(k_cache).copy()
    vc8 = _u8(v_cache).copy()
    shape = kc8.shape
    runs = []
    for fill in (0x0000, 0xFFFF):
        scratch = np.full(shape, fill, dtype=np.uint16)
        runs.append(qk_norm_rope_write(
            qkv, q_norm_w, k_norm_w, scratch, scratch, block_table, context_lens, chunk_lens,
            num_q_heads, num_kv_heads, num_pages, max_pages_per_seq, eps=eps,
            rope_base=rope_base, rope_scale=rope_scale, q_scale=q_scale, page_size=page_size,
            head_dim=head_dim))
    (q_out, k0, v0, skipped), (_, k1, v1, _) = runs
    written = np.all(k0 == k1, axis=(-2, -1)) & np.all(v0 == v1, axis=(-2, -1))
    ks = np.ascontiguousarray(k_scale, dtype=np.float32)[None, :, None]
    vs = np.ascontiguousarray(v_scale, dtype=np.float32)[None, :, None]
    for src, scl, dst in ((k0, ks, kc8), (v0, vs, vc8)):
        rows = (src[written].astype(np.uint32) << 16).view(np.float32)  # exact bf16 values
        dst[written] = e4m3_encode((rows / scl).astype(np.float32))
    return q_out, kc8, vc8, skipped


def topk(logits, k):
    """Exact top-k of each row of logits [rows, vocab] (float32): values and int32
    indices [rows, k], larger first, NaN above +inf, ties by smaller index."""
    x = np.ascontiguousarray(logits, dtype=np.float32)
    rows, vocab = x.shape
    vals = np.zeros((max(rows, 1), k), dtype=np.float32)
    idx = np.zeros((max(rows, 1), k), dtype=np.int32)
    _load().oracle_topk(x, vocab, rows, vocab, int(k), vals, idx)
    return vals[:rows], idx[:rows]
