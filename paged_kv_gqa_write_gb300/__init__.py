"""Python binding of libpagedattn.so -- paged-KV GQA attention for GB300.

Thin ctypes marshalling over the C ABI declared in ``include/pagedattn.h``:
the functions here have the C entry points' names, derive ``pa_dims`` from
tensor shapes, check dtypes/devices, pass raw device pointers and the current
CUDA stream, and raise on a non-zero return code.  Every step of the path runs
in the library's CUDA kernels; there is no fallback.  PyTorch supplies device
memory and streams only.
"""
import ctypes
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpagedattn.so")

HEAD_DIM = 128
PAGE_SIZE = 128
PA_BF16, PA_F32 = 0, 1
PA_STATUS_BAD_PAGE, PA_STATUS_BAD_LENGTH, PA_STATUS_BAD_TOKENS, PA_STATUS_TIMEOUT = 1, 2, 4, 8
PA_STATUS_Q_RANGE = 16
PA_MAX_CHUNKED_SEQS = 16384
PA_SPLITS_BALANCED = -1
PA_BALANCED_MAX_SEQS = 512
PA_TOPK_MAX_K = 32
PA_MAX_Q_LEN = 16
PA_MAX_PROLOGUE_HEADS = 384
PA_PREFILL_SCHEDULE_ITEMS = 64
(PA_ERR_NULL_POINTER, PA_ERR_HEAD_DIM, PA_ERR_PAGE_SIZE, PA_ERR_HEADS, PA_ERR_DIMS,
 PA_ERR_ALIGNMENT, PA_ERR_OUT_DTYPE, PA_ERR_WORKSPACE, PA_ERR_SPLITS, PA_ERR_TOO_MANY_SEQS,
 PA_ERR_TENSOR_MAP, PA_ERR_NO_DEVICE, PA_ERR_NOALLOC_TOO_LARGE) = range(-1, -14, -1)

EXPORTED = ("pa_kv_write", "pa_decode", "pa_decode_workspace_size", "pa_decode_auto_splits",
            "pa_prefill_chunk", "pa_combine", "pa_status_string", "pa_abi_version",
            "pa_decode_noalloc", "pa_qk_norm_rope_write", "pa_topk", "pa_topk_workspace_size",
            "pa_decode_multi", "pa_decode_multi_workspace_size", "pa_kv_write_fp8",
            "pa_decode_fp8", "pa_wait_selftest", "pa_prefill_pairs", "pa_prefill_chunk_fp8",
            "pa_qk_norm_rope_write_fp8", "pa_decode_prologue")
PA_NOALLOC_SCRATCH_BYTES = 16 << 20


class pa_dims(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("num_pages", ctypes.c_int32),
                ("max_pages_per_seq", ctypes.c_int32)]


class PagedAttnError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn} failed: {code} ({pa_status_string(code)})")
        self.code = code


_lib = None


def load(path: str = LIB_PATH):
    """Load the CUDA library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -c \"import __graft_entry__ as g; "
                           f"g.build()\"` (there is no non-CUDA path)")
    lib = ctypes.CDLL(path)
    vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
    lib.pa_kv_write.restype = ctypes.c_int
    lib.pa_kv_write.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, pa_dims, vp, vp]
    lib.pa_qk_norm_rope_write.restype = ctypes.c_int
    lib.pa_qk_norm_rope_write.argtypes = [vp, vp, vp, f32, f32, f32, f32, vp, vp, vp, vp, vp,
                                          vp, i32, pa_dims, vp, vp]
    lib.pa_qk_norm_rope_write_fp8.restype = ctypes.c_int
    lib.pa_qk_norm_rope_write_fp8.argtypes = [vp, vp, vp, f32, f32, f32, f32, vp, vp, vp, vp, vp,
                                              vp, vp, vp, i32, pa_dims, vp, vp]
    lib.pa_decode_prologue.restype = ctypes.c_int
    lib.pa_decode_prologue.argtypes = [vp, vp, vp, f32, f32, f32, f32, vp, vp, vp, vp, f32, vp,
                                       i32, vp, sz, i32, pa_dims, vp, vp]
    lib.pa_topk.restype = ctypes.c_int
    lib.pa_topk.argtypes = [vp, ctypes.c_int64, i32, i32, i32, vp, vp, vp, sz, vp]
    lib.pa_topk_workspace_size.restype = sz
    lib.pa_topk_workspace_size.argtypes = [i32, i32, i32]
    lib.pa_decode.restype = ctypes.c_int
    lib.pa_decode.argtypes = [vp, vp, vp, vp, vp, f32, vp, i32, vp, sz, i32, pa_dims, vp, vp]
    lib.pa_decode_multi.restype = ctypes.c_int
    lib.pa_decode_multi.argtypes = [vp, vp, vp, vp, vp, i32, f32, vp, i32, vp, sz, i32, pa_dims,
                                    vp, vp]
    lib.pa_kv_write_fp8.restype = ctypes.c_int
    lib.pa_kv_write_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, pa_dims, vp, vp]
    lib.pa_decode_fp8.restype = ctypes.c_int
    lib.pa_decode_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, f32, vp, i32, vp, sz, i32,
                                  pa_dims, vp, vp]
    lib.pa_decode_multi_workspace_size.restype = sz
    lib.pa_decode_multi_workspace_size.argtypes = [pa_dims, i32, i32]
    lib.pa_decode_workspace_size.restype = sz
    lib.pa_decode_workspace_size.argtypes = [pa_dims, i32]
    lib.pa_decode_auto_splits.restype = i32
    lib.pa_decode_auto_splits.argtypes = [pa_dims]
    lib.pa_prefill_chunk.restype = ctypes.c_int
    lib.pa_prefill_chunk.argtypes = [vp, vp, vp, vp, vp, vp, i32, f32, vp, i32, pa_dims, vp, vp]
    lib.pa_prefill_chunk_fp8.restype = ctypes.c_int
    lib.pa_prefill_chunk_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, f32, vp, i32,
                                         pa_dims, vp, vp]
    lib.pa_combine.restype = ctypes.c_int
    lib.pa_combine.argtypes = [vp, vp, i32, vp, i32, pa_dims, vp]
    lib.pa_decode_noalloc.restype = ctypes.c_int
    lib.pa_decode_noalloc.argtypes = [vp, vp, vp, vp, vp, f32, vp, i32, i32, pa_dims, vp, vp]
    lib.pa_prefill_pairs.restype = i32
    lib.pa_prefill_pairs.argtypes = []
    lib.pa_wait_selftest.restype = ctypes.c_int
    lib.pa_wait_selftest.argtypes = [ctypes.c_uint32, vp, vp]
    lib.pa_status_string.restype = ctypes.c_char_p
    lib.pa_status_string.argtypes = [i32]
    lib.pa_abi_version.restype = i32
    lib.pa_abi_version.argtypes = []
    _lib = lib
    return lib


def pa_status_string(code: int) -> str:
    return load().pa_status_string(int(code)).decode()


def pa_abi_version() -> int:
    return int(load().pa_abi_version())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(fn, rc):
    if rc != 0:
        raise PagedAttnError(fn, rc)


def _need(t, name, dtype, device=None):
    if t is None:
        raise ValueError(f"{name} is required")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def make_dims(num_seqs, num_q_heads, num_kv_heads, num_pages, max_pages_per_seq):
    return pa_dims(int(num_seqs), int(num_q_heads), int(num_kv_heads), HEAD_DIM, PAGE_SIZE,
                   int(num_pages), int(max_pages_per_seq))


def _cache_dims(q_heads, k_cache, block_table):
    num_pages, page, hkv, d = k_cache.shape
    if page != PAGE_SIZE or d != HEAD_DIM:
        raise ValueError(f"cache must be [pages, {PAGE_SIZE}, Hkv, {HEAD_DIM}], got {tuple(k_cache.shape)}")
    return make_dims(block_table.shape[0], q_heads, hkv, num_pages, block_table.shape[1])


def pa_kv_write(k_new, v_new, k_cache, v_cache, block_table, context_lens, chunk_lens=None,
                status=None, stream=None):
    """Write new tokens' K/V ([T, Hkv, 128] bf16) into the paged caches in place."""
    dev = k_cache.device
    for t, n in ((k_new, "k_new"), (v_new, "v_new"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, torch.bfloat16, dev)
    _need(block_table, "block_table", torch.int32, dev)
    _need(context_lens, "context_lens", torch.int32, dev)
    if chunk_lens is not None:
        _need(chunk_lens, "chunk_lens", torch.int32, dev)
    if status is not None:
        _need(status, "status", torch.int32, dev)
    d = _cache_dims(k_cache.shape[2], k_cache, block_table)
    rc = load().pa_kv_write(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                            _ptr(block_table), _ptr(context_lens), _ptr(chunk_lens),
                            int(k_new.shape[0]), d, _ptr(status), _stream(stream))
    _check("pa_kv_write", rc)


def pa_qk_norm_rope_write(qkv, q_norm_w, k_norm_w, k_cache, v_cache, block_table,
                          context_lens, chunk_lens=None, eps=1e-6, rope_base=1e6,
                          rope_scale=1.0, q_scale=1.0, q_out=None, status=None, stream=None):
    """Q/K RMSNorm -> NeoX RoPE -> KV cache write for the new tokens.  qkv is the
    fused projection output [T, (Hq + 2 Hkv) * 128] bf16; returns q_out [T, Hq, 128]."""
    dev = k_cache.device
    _need(qkv, "qkv", torch.bfloat16, dev)
    _need(k_cache, "k_cache", torch.bfloat16, dev)
    _need(v_cache, "v_cache", torch.bfloat16, dev)
    _need(q_norm_w, "q_norm_w", torch.float32, dev)
    _need(k_norm_w, "k_norm_w", torch.float32, dev)
    _need(block_table, "block_table", torch.int32, dev)
    _need(context_lens, "context_lens", torch.int32, dev)
    if chunk_lens is not None:
        _need(chunk_lens, "chunk_lens", torch.int32, dev)
    if status is not None:
        _need(status, "status", torch.int32, dev)
    Hkv = k_cache.shape[2]
    T = qkv.shape[0]
    Hq = qkv.reshape(T, -1).shape[1] // HEAD_DIM - 2 * Hkv
    d = _cache_dims(Hq, k_cache, block_table)
    if q_out is None:
        q_out = torch.empty(T, Hq, HEAD_DIM, dtype=torch.bfloat16, device=dev)
    _need(q_out, "q_out", torch.bfloat16, dev)
    rc = load().pa_qk_norm_rope_write(
        _ptr(qkv), _ptr(q_norm_w), _ptr(k_norm_w), float(eps), float(rope_base),
        float(rope_scale), float(q_scale), _ptr(q_out), _ptr(k_cache), _ptr(v_cache),
        _ptr(block_table), _ptr(context_lens), _ptr(chunk_lens), int(T), d, _ptr(status),
        _stream(stream))
    _check("pa_qk_norm_rope_write", rc)
    return q_out


def pa_qk_norm_rope_write_fp8(qkv, q_norm_w, k_norm_w, k_cache, v_cache, k_scale, v_scale,
                              block_table, context_lens, chunk_lens=None, eps=1e-6,
                              rope_base=1e6, rope_scale=1.0, q_scale=1.0, q_out=None,
                              status=None, stream=None):
    """The prologue into an FP8 (e4m3) cache [num_pages, 128, Hkv, 128] with
    per-KV-head float32 scales; returns q_out [T, Hq, 128] bf16."""
    dev = k_cache.device
    _need(qkv, "qkv", torch.bfloat16, dev)
    _need_fp8_cache(k_cache, "k_cache", dev)
    _need_fp8_cache(v_cache, "v_cache", dev)
    _need(k_scale, "k_scale", torch.float32, dev)
    _need(v_scale, "v_scale", torch.float32, dev)
    _need(q_norm_w, "q_norm_w", torch.float32, dev)
    _need(k_norm_w, "k_norm_w", torch.float32, dev)
    _need(block_table, "block_table", torch.int32, dev)
    _need(context_lens, "context_lens", torch.int32, dev)
    if chunk_lens is not None:
        _need(chunk_lens, "chunk_lens", torch.int32, dev)
    if status is not None:
        _need(status, "status", torch.int32, dev)
    Hkv = k_cache.shape[2]
    T = qkv.shape[0]
    Hq = qkv.reshape(T, -1).shape[1] // HEAD_DIM - 2 * Hkv
    d = _cache_dims(Hq, k_cache, block_table)
    if q_out is None:
        q_out = torch.empty(T, Hq, HEAD_DIM, dtype=torch.bfloat16, device=dev)
    _need(q_out, "q_out", torch.bfloat16, dev)
    rc = load().pa_qk_norm_rope_write_fp8(
        _ptr(qkv), _ptr(q_norm_w), _ptr(k_norm_w), float(eps), float(rope_base),
        float(rope_scale), float(q_scale), _ptr(q_out), _ptr(k_cache), _ptr(v_cache),
        _ptr(k_scale), _ptr(v_scale), _ptr(block_table), _ptr(context_lens), _ptr(chunk_lens),
        int(T), d, _ptr(status), _stream(stream))
    _check("pa_qk_norm_rope_write_fp8", rc)
    return q_out


def pa_topk(logits, k, out_values=None, out_indices=None, workspace=None, stream=None):
    """Exact top-k of each row of logits [rows, vocab] float32 (row stride may
    exceed vocab).  Returns (values [rows, k] float32, indices [rows, k] int32)."""
    dev = logits.device
    if logits.dtype != torch.float32 or logits.dim() != 2 or logits.stride(1) != 1:
        raise TypeError("logits must be a float32 [rows, vocab] tensor with unit column stride")
    rows, vocab = logits.shape
    if out_values is None:
        out_values = torch.empty(rows, k, dtype=torch.float32, device=dev)
    if out_indices is None:
        out_indices = torch.empty(rows, k, dtype=torch.int32, device=dev)
    need = int(load().pa_topk_workspace_size(rows, vocab, int(k)))
    if need == (1 << 64) - 1:
        raise ValueError("unsupported rows / vocab / k for pa_topk")
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    rc = load().pa_topk(_ptr(logits), int(logits.stride(0)), int(rows), int(vocab), int(k),
                        _ptr(out_values), _ptr(out_indices), _ptr(workspace),
                        workspace.numel() * workspace.element_size(), _stream(stream))
    _check("pa_topk", rc)
    return out_values, out_indices


def pa_decode_workspace_size(dims, num_splits=0) -> int:
    n = int(load().pa_decode_workspace_size(dims, int(num_splits)))
    if n == (1 << 64) - 1:
        raise ValueError("invalid dims or schedule for pa_decode_workspace_size")
    return n


def pa_decode_auto_splits(dims) -> int:
    r = int(load().pa_decode_auto_splits(dims))
    if r < 0:
        raise PagedAttnError("pa_decode_auto_splits", r)
    return r


def pa_decode(q, k_cache, v_cache, block_table, context_lens, scale=None, out=None,
              out_dtype=torch.bfloat16, workspace=None, num_splits=0, status=None, stream=None):
    """Single-token paged GQA decode.  q: [B, Hq, 128] bf16.  Returns out [B, Hq, 128]."""
    dev = k_cache.device
    _need(q, "q", torch.bfloat16, dev)
    _need(k_cache, "k_cache", torch.bfloat16, dev)
    _need(v_cache, "v_cache", torch.bfloat16, dev)
    _need(block_table, "block_table", torch.int32, dev)
    _need(context_lens, "context_lens", torch.int32, dev)
    if status is not None:
        _need(status, "status", torch.int32, dev)
    B, Hq, D = q.shape
    d = _cache_dims(Hq, k_cache, block_table)
    if out is None:
        out = torch.empty(B, Hq, D, dtype=out_dtype, device=dev)
    _need(out, "out", out.dtype, dev)
    code = PA_F32 if out.dtype == torch.float32 else PA_BF16
    if out.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("out must be bf16 or f32")
    need = pa_decode_workspace_size(d, num_splits)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    rc = load().pa_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                          _ptr(context_lens), scale, _ptr(out), code, _ptr(workspace),
                          0 if workspace is None else workspace.numel() * workspace.element_size(),
                          int(num_splits), d, _ptr(status), _stream(stream))
    _check("pa_decode", rc)
    return out


def pa_decode_prologue(qkv, q_norm_w, k_norm_w, k_cache, v_cache, block_table, context_lens,
                       eps=1e-6, rope_base=1e6, rope_scale=1.0, q_scale=1.0, scale=None,
                       out=None, out_dtype=torch.bfloat16, workspace=None, num_splits=0,
                       status=None, stream=None):
    """The decode step with its prologue in the attention kernel: qkv is the fused
    projection output [B, (Hq + 2 Hkv) * 128] bf16 (one new token per sequence);
    writes the new tokens' K/V rows into the caches and returns out [B, Hq, 128].
    Equal to pa_qk_norm_rope_write followed by pa_decode."""
    dev = k_cache.device
    _need(qkv, "qkv", torch.bfloat16, dev)
    _need(q_norm_w, "q_norm_w", torch.float32, dev)
    _need(k_norm_w, "k_norm_w", torch.float32, dev)
    _need(k_cache, "k_cache", torch.bfloat16, dev)
    _need(v_cache, "v_cache", torch.bfloat16, dev)
    _need(block_table, "block_table", torch.int32, dev)
    _need(context_lens, "context_lens", torch.int32, dev)
    if status is not None:
        _need(status, "status", torch.int32, dev)
    B = qkv.shape[0]
    Hkv = k_cache.shape[2]
    Hq = qkv.reshape(B, -1).shape[1] // HEAD_DIM - 2 * Hkv
    d = _cache_dims(Hq, k_cache, block_table)
    if B != d.num_seqs:
        raise ValueError(f"qkv has {B} rows; expected one per sequence ({d.num_seqs})")
    if out is None:
        out = torch.empty(B, Hq, HEAD_DIM, dtype=out_dtype, device=dev)
    if out.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("out must be bf16 or f32")
    _need(out, "out", out.dtype, dev)
    code = PA_F32 if out.dtype == torch.float32 else PA_BF16
    need = pa_decode_workspace_size(d, num_splits)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    scale = 1.0 / math.sqrt(HEAD_DIM) if scale is None else float(scale)
    rc = load().pa_decode_prologue(
        _ptr(qkv), _ptr(q_norm_w), _ptr(k_norm_w), float(eps), float(rope_base),
        float(rope_scale), float(q_scale), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
        _ptr(context_lens), scale, _ptr(out), code, _ptr(workspace),
        0 if workspace is None else workspace.numel() * workspace.element_size(),
        int(num_splits), d, _ptr(status), _stream(stream))
    _check("pa_decode_prologue", rc)
    return out


def pa_decode_multi_workspace_size(dims, q_len, num_splits=0) -> int:
    n = int(load().pa_decode_multi_workspace_size(dims, int(q_len), int(num_splits)))
    if n == (1 << 64) - 1:
        raise ValueError("invalid dims, q_len or schedule for pa_decode_multi_workspace_size")
    return n


def pa_decode_multi(q, k_cache, v_cache, block_table, context_lens, q_len, scale=None, out=None,
                    out_dtype=torch.bfloat16, workspace=None, num_splits=0, status=None,
                    stream=None):
    """Multi-token decode: q_len new tokens per sequence, q [B * q_len, Hq, 128] bf16
    token-major; token j of sequence s attends to keys 0 .. context_lens[s] - q_len + j.
    Returns out [B * q_len, Hq, 128]."""
    dev = k_cache.device
    _need(q, "q", torch.bfloat16, dev)
    _need(k_cache, "k_cache", torch.bfloat16, dev)
    _need(v_cache, "v_cache", torch.bfloat16, dev)
    _need(block_table, "block_table", torch.int32, dev)
    _need(context_lens, "context_lens", torch.int32, dev)
    if status is not None:
        _need(status, "status", torch.int32, dev)
    T, Hq, D = q.shape
    d = _cache_dims(Hq, k_cache, block_table)
    q_len = int(q_len)
    if q_len < 1 or T != d.num_seqs * q_len:
        raise ValueError(f"q has {T} rows; expected num_seqs ({d.num_seqs}) x q_len ({q_len})")
    if out is None:
        out = torch.empty(T, Hq, D, dtype=out_dtype, device=dev)
    _need(out, "out", out.dtype, dev)
    if out.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("out must be bf16 or f32")
    code = PA_F32 if out.dtype == torch.float32 else PA_BF16
    need = pa_decode_multi_workspace_size(d, q_len, num_splits)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().pa_decode_multi(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                                _ptr(context_lens), q_len, scale, _ptr(out), code,
                                _ptr(workspace), ws_bytes, int(num_splits), d, _ptr(status),
                                _stream(stream))
    _check("pa_decode_multi", rc)
    return out


def _need_fp8_cache(t, name, dev):
    if t.device != dev or t.dtype not in (torch.uint8, getattr(torch, "float8_e4m3fn", None)):
        raise TypeError(f"{name} must be a uint8 (or float8_e4m3fn) tensor on {dev}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def pa_kv_write_fp8(k_new, v_new, k_cache, v_cache, k_scale, v_scale, block_table, context_lens,
                    chunk_lens=None, status=None, stream=None):
    """Quantizing KV write into an FP8 (e4m3) cache [num_pages, 128, Hkv, 128] with
    per-KV-head float32 scales."""
    dev = k_cache.device
    _need(k_new, "k_new", torch.bfloat16, dev)
    _need(v_new, "v_new", torch.bfloat16, dev)
    _need_fp8_cache(k_cache, "k_cache", dev)
    _need_fp8_cache(v_cache, "v_cache", dev)
    _need(k_scale, "k_scale", torch.float32, dev)
    _need(v_scale, "v_scale", torch.float32, dev)
    _need(block_table, "block_table", torch.int32, dev)
    _need(context_lens, "context_lens", torch.int32, dev)
    if chunk_lens is not None:
        _need(chunk_lens, "chunk_lens", torch.int32, dev)
    if status is not None:
        _need(status, "status", torch.int32, dev)
    T = k_new.shape[0]
    d = _cache_dims(k_cache.shape[2], k_cache, block_table)
    rc = load().pa_kv_write_fp8(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                _ptr(k_scale), _ptr(v_scale), _ptr(block_table),
                                _ptr(context_lens), _ptr(chunk_lens), T, d, _ptr(status),
                                _stream(stream))
    _check("pa_kv_write_fp8", rc)


def pa_decode_fp8(q, k_cache, v_cache, k_scale, v_scale, block_table, context_lens, q_len=1,
                  scale=None, out=None, out_dtype=torch.bfloat16, workspace=None, num_splits=0,
                  status=None, stream=None):
    """Decode (q_len new tokens per sequence) over an FP8 (e4m3) cache with
    per-KV-head scales.  q: [B * q_len, Hq, 128] bf16.  Returns out [B * q_len, Hq, 128]."""
    dev = k_cache.device
    _need(q, "q", torch.bfloat16, dev)
    _need_fp8_cache(k_cache, "k_cache", dev)
    _need_fp8_cache(v_cache, "v_cache", dev)
    _need(k_scale, "k_scale", torch.float32, dev)
    _need(v_scale, "v_scale", torch.float32, dev)
    _need(block_table, "block_table", torch.int32, dev)
    _need(context_lens, "context_lens", torch.int32, dev)
    if status is not None:
        _need(status, "status", torch.int32, dev)
    T, Hq, D = q.shape
    d = _cache_dims(Hq, k_cache, block_table)
    q_len = int(q_len)
    if q_len < 1 or T != d.num_seqs * q_len:
        raise ValueError(f"q has {T} rows; expected num_seqs ({d.num_seqs}) x q_len ({q_len})")
    if out is None:
        out = torch.empty(T, Hq, D, dtype=out_dtype, device=dev)
    _need(out, "out", out.dtype, dev)
    if out.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("out must be bf16 or f32")
    code = PA_F32 if out.dtype == torch.float32 else PA_BF16
    need = pa_decode_multi_workspace_size(d, q_len, num_splits)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().pa_decode_fp8(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
                              _ptr(v_scale), _ptr(block_table), _ptr(context_lens), q_len, scale,
                              _ptr(out), code, _ptr(workspace), ws_bytes, int(num_splits), d,
                              _ptr(status), _stream(stream))
    _check("pa_decode_fp8", rc)
    return out


def pa_prefill_chunk(q, k_cache, v_cache, block_table, context_lens, chunk_lens, scale=None,
                     out=None, out_dtype=torch.bfloat16, status=None, stream=None):
    """Causal chunked prefill over the paged cache.  q: [T, Hq, 128] bf16 token-major."""
    dev = k_cache.device
    _need(q, "q", torch.bfloat16, dev)
    _need(k_cache, "k_cache", torch.bfloat16, dev)
    _need(v_cache, "v_cache", torch.bfloat16, dev)
    _need(block_table, "block_table", torch.int32, dev)
    _need(context_lens, "context_lens", torch.int32, dev)
    _need(chunk_lens, "chunk_lens", torch.int32, dev)
    if status is not None:
        _need(status, "status", torch.int32, dev)
    T, Hq, D = q.shape
    d = _cache_dims(Hq, k_cache, block_table)
    if out is None:
        out = torch.empty(T, Hq, D, dtype=out_dtype, device=dev)
    _need(out, "out", out.dtype, dev)
    if out.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("out must be bf16 or f32")
    code = PA_F32 if out.dtype == torch.float32 else PA_BF16
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    rc = load().pa_prefill_chunk(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                                 _ptr(context_lens), _ptr(chunk_lens), int(T), scale, _ptr(out),
                                 code, d, _ptr(status), _stream(stream))
    _check("pa_prefill_chunk", rc)
    return out


def pa_prefill_chunk_fp8(q, k_cache, v_cache, k_scale, v_scale, block_table, context_lens,
                         chunk_lens, scale=None, out=None, out_dtype=torch.bfloat16, status=None,
                         stream=None):
    """Causal chunked prefill over an FP8 (e4m3) cache [num_pages, 128, Hkv, 128] with
    per-KV-head float32 scales.  q: [T, Hq, 128] bf16 token-major."""
    dev = k_cache.device
    _need(q, "q", torch.bfloat16, dev)
    _need_fp8_cache(k_cache, "k_cache", dev)
    _need_fp8_cache(v_cache, "v_cache", dev)
    _need(k_scale, "k_scale", torch.float32, dev)
    _need(v_scale, "v_scale", torch.float32, dev)
    _need(block_table, "block_table", torch.int32, dev)
    _need(context_lens, "context_lens", torch.int32, dev)
    _need(chunk_lens, "chunk_lens", torch.int32, dev)
    if status is not None:
        _need(status, "status", torch.int32, dev)
    T, Hq, D = q.shape
    d = _cache_dims(Hq, k_cache, block_table)
    if out is None:
        out = torch.empty(T, Hq, D, dtype=out_dtype, device=dev)
    _need(out, "out", out.dtype, dev)
    if out.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("out must be bf16 or f32")
    code = PA_F32 if out.dtype == torch.float32 else PA_BF16
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    rc = load().pa_prefill_chunk_fp8(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
                                     _ptr(v_scale), _ptr(block_table), _ptr(context_lens),
                                     _ptr(chunk_lens), int(T), scale, _ptr(out), code, d,
                                     _ptr(status), _stream(stream))
    _check("pa_prefill_chunk_fp8", rc)
    return out


def pa_combine(part_o, part_lse, out=None, out_dtype=torch.float32, stream=None):
    """Merge partial states part_o [B, Hq, S, 128] f32 / part_lse [B, Hq, S] f32."""
    dev = part_o.device
    _need(part_o, "part_o", torch.float32, dev)
    _need(part_lse, "part_lse", torch.float32, dev)
    B, Hq, S, D = part_o.shape
    if out is None:
        out = torch.empty(B, Hq, D, dtype=out_dtype, device=dev)
    _need(out, "out", out.dtype, dev)
    code = PA_F32 if out.dtype == torch.float32 else PA_BF16
    d = make_dims(B, Hq, 1, 1, 1)
    rc = load().pa_combine(_ptr(part_o), _ptr(part_lse), int(S), _ptr(out), code, d,
                           _stream(stream))
    _check("pa_combine", rc)
    return out


def pa_decode_noalloc(q, k_cache, v_cache, block_table, context_lens, scale=None, out=None,
                      out_dtype=torch.bfloat16, num_splits=0, status=None, stream=None):
    """pa_decode without a workspace, for callers that cannot allocate device
    memory: the split partials go to the library's fixed device array
    (PA_NOALLOC_SCRATCH_BYTES).  Calls on one device share that array, so calls
    that may overlap on the GPU must be ordered on one stream.  `out` should be
    passed in by such callers (allocating it here is a convenience)."""
    dev = k_cache.device
    _need(q, "q", torch.bfloat16, dev)
    _need(k_cache, "k_cache", torch.bfloat16, dev)
    _need(v_cache, "v_cache", torch.bfloat16, dev)
    _need(block_table, "block_table", torch.int32, dev)
    _need(context_lens, "context_lens", torch.int32, dev)
    if status is not None:
        _need(status, "status", torch.int32, dev)
    B, Hq, D = q.shape
    d = _cache_dims(Hq, k_cache, block_table)
    if out is None:
        out = torch.empty(B, Hq, D, dtype=out_dtype, device=dev)
    _need(out, "out", out.dtype, dev)
    if out.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("out must be bf16 or f32")
    code = PA_F32 if out.dtype == torch.float32 else PA_BF16
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    rc = load().pa_decode_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                                  _ptr(context_lens), scale, _ptr(out), code, int(num_splits), d,
                                  _ptr(status), _stream(stream))
    _check("pa_decode_noalloc", rc)
    return out


def pa_wait_selftest(limit_us=2000, status=None, stream=None):
    """Run the kernels' bounded-wait failure path once: a wait on an mbarrier
    that nothing arrives on gives up after limit_us and sets PA_STATUS_TIMEOUT
    in `status` (a 1-element int32 device tensor, created when omitted).
    Returns `status`."""
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
    _need(status, "status", torch.int32, status.device)
    rc = load().pa_wait_selftest(int(limit_us), _ptr(status), _stream(stream))
    _check("pa_wait_selftest", rc)
    return status


def pa_prefill_pairs() -> int:
    """CTA pairs a pa_prefill_chunk launch uses at most on the current device."""
    n = int(load().pa_prefill_pairs())
    if n < 1:
        raise PagedAttnError("pa_prefill_pairs", n)
    return n
