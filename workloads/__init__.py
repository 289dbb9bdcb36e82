"""Seeded synthetic inputs for the paged-KV GQA attention path.

This module builds inputs only: page pools, block tables, lengths and the
query / new-token tensors, all drawn from seeded generators.  It holds none of
the attention arithmetic, so both the CUDA path's tests and the CPU oracle can
consume the same bits.

Recipe (shapes from the "Qwen3-14B" pypto-lib doc, "Deployment configuration":
40 query heads over 8 KV heads, head_dim 128, contexts up to 4096 in 128-token
pages, decode padded to 16 rows; Qwen3-32B uses 64 query heads over 8):
  * values: N(0, 1) float32 from a seeded ``torch.Generator``, rounded to
    bfloat16 (round-to-nearest-even); seed = config index * 1000 + tensor id;
  * K/V cache: [num_pages, 128, Hkv, 128] bfloat16 (vLLM order);
  * poison: every pool page no sequence references, the tail slots past each
    sequence's context in its last page, and the slots a KV write is about to
    fill are set to NaN, so any stray read shows up in the output;
  * block tables: int32 [B, max_pages_per_seq], unused entries -1.
"""
from dataclasses import dataclass, field
import math
from typing import List, Optional

import torch

PAGE = 128
HEAD_DIM = 128
NAN_BF16 = 0x7FC0

# tensor ids inside a config's seed space
_T_K, _T_V, _T_Q, _T_KNEW, _T_VNEW, _T_LEN, _T_PERM, _T_PRIOR = 1, 2, 3, 4, 5, 6, 7, 8
_T_QKV, _T_WQ, _T_WK = 9, 10, 11


@dataclass
class PagedCase:
    name: str
    B: int
    Hq: int
    Hkv: int
    num_pages: int
    max_pages_per_seq: int
    q: torch.Tensor                 # bf16 [T, Hq, D]
    k_cache: torch.Tensor           # bf16 [num_pages, PAGE, Hkv, D]
    v_cache: torch.Tensor
    block_table: torch.Tensor       # int32 [B, max_pages_per_seq]
    context_lens: torch.Tensor      # int32 [B], length after the write
    chunk_lens: Optional[torch.Tensor] = None  # int32 [B]; None = decode (1 per seq)
    k_new: Optional[torch.Tensor] = None       # bf16 [T, Hkv, D]
    v_new: Optional[torch.Tensor] = None
    scale: float = 1.0 / math.sqrt(HEAD_DIM)
    poisoned_pages: List[int] = field(default_factory=list)

    @property
    def T(self) -> int:
        return self.B if self.chunk_lens is None else int(self.chunk_lens.sum())

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    def to(self, device) -> "PagedCase":
        out = PagedCase(**{k: getattr(self, k) for k in self.__dataclass_fields__})
        for k in ("q", "k_cache", "v_cache", "block_table", "context_lens", "chunk_lens",
                  "k_new", "v_new"):
            v = getattr(out, k)
            if v is not None:
                setattr(out, k, v.to(device))
        return out


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def randn_bf16(shape, seed: int, device="cpu", chunk_rows: int = 1 << 22) -> torch.Tensor:
    """N(0,1) float32 rounded to bfloat16, generated in chunks along dim 0 with one
    seeded generator (deterministic for a given device kind)."""
    shape = tuple(shape)
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    if out.numel() == 0:
        return out
    g = _gen(seed, device)
    flat = out.view(-1)
    n = flat.numel()
    for i in range(0, n, chunk_rows):
        m = min(chunk_rows, n - i)
        flat[i:i + m] = torch.randn(m, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    return out


def _poison_pages(cache: torch.Tensor, pages) -> None:
    if len(pages):
        idx = torch.as_tensor(list(pages), dtype=torch.long, device=cache.device)
        cache.view(torch.int16)[idx] = NAN_BF16


def _poison_slots(cache: torch.Tensor, slots) -> None:
    if len(slots):
        idx = torch.as_tensor(list(slots), dtype=torch.long, device=cache.device)
        flat = cache.view(torch.int16).view(-1, PAGE, cache.shape[2], cache.shape[3])
        flat.view(-1, cache.shape[2], cache.shape[3])[idx] = NAN_BF16


def build_case(name: str, seed_base: int, ctx_lens, Hq: int, Hkv: int, num_pages: int,
               page_lists, max_pages_per_seq: int, chunk_lens=None, with_new: bool = False,
               device="cpu", poison: bool = True, pool_device=None) -> PagedCase:
    """Assemble a case from explicit lengths and per-sequence physical page lists.

    ctx_lens: length of each sequence after the write; chunk_lens: new tokens per
    sequence (None = decode, one query per sequence).  with_new: also draw the new
    tokens' K/V (k_new, v_new) and poison the slots they will be written to."""
    B = len(ctx_lens)
    ctx = torch.tensor(ctx_lens, dtype=torch.int32)
    cl = None if chunk_lens is None else torch.tensor(chunk_lens, dtype=torch.int32)
    n_new = [1] * B if cl is None else list(chunk_lens)
    T = sum(n_new) if cl is not None else B
    bt = torch.full((B, max_pages_per_seq), -1, dtype=torch.int32)
    used = set()
    for s in range(B):
        need = (ctx_lens[s] + PAGE - 1) // PAGE
        assert len(page_lists[s]) >= need, (s, need, len(page_lists[s]))
        assert need <= max_pages_per_seq
        for i in range(need):
            bt[s, i] = int(page_lists[s][i])
            used.add(int(page_lists[s][i]))
    pdev = pool_device or device
    k_cache = randn_bf16((num_pages, PAGE, Hkv, HEAD_DIM), seed_base + _T_K, pdev)
    v_cache = randn_bf16((num_pages, PAGE, Hkv, HEAD_DIM), seed_base + _T_V, pdev)
    q = randn_bf16((T, Hq, HEAD_DIM), seed_base + _T_Q, device)
    k_new = v_new = None
    if with_new:
        k_new = randn_bf16((T, Hkv, HEAD_DIM), seed_base + _T_KNEW, device)
        v_new = randn_bf16((T, Hkv, HEAD_DIM), seed_base + _T_VNEW, device)
    poisoned = []
    if poison:
        poisoned = sorted(set(range(num_pages)) - used)
        tails = []
        for s in range(B):
            c = ctx_lens[s]
            if c % PAGE:
                last = int(bt[s, (c - 1) // PAGE])
                tails += [last * PAGE + t for t in range(c % PAGE, PAGE)]
            if with_new:
                for j in range(n_new[s]):
                    pos = c - n_new[s] + j
                    tails.append(int(bt[s, pos // PAGE]) * PAGE + pos % PAGE)
        for cache in (k_cache, v_cache):
            _poison_pages(cache, poisoned)
            _poison_slots(cache, tails)
    return PagedCase(name=name, B=B, Hq=Hq, Hkv=Hkv, num_pages=num_pages,
                     max_pages_per_seq=max_pages_per_seq, q=q, k_cache=k_cache,
                     v_cache=v_cache, block_table=bt.to(device), context_lens=ctx.to(device),
                     chunk_lens=None if cl is None else cl.to(device), k_new=k_new, v_new=v_new,
                     poisoned_pages=poisoned)


def _perm(n: int, seed: int) -> List[int]:
    return torch.randperm(n, generator=_gen(seed)).tolist()


def consecutive_runs(ctx_lens, perm) -> List[List[int]]:
    """Sequence s takes the next ceil(ctx/128) entries of the permutation."""
    out, i = [], 0
    for c in ctx_lens:
        need = (c + PAGE - 1) // PAGE
        out.append(perm[i:i + need])
        i += need
    assert i <= len(perm)
    return out


# ---------------------------------------------------------------- the five workloads

def tiny_decode(device="cpu", with_new=False) -> PagedCase:
    """batch 2, 8 Q heads over 2 KV heads, contexts {1, 200}, a 4-page pool assigned
    by a seeded permutation (seq 0: 1 page, seq 1: 2 pages, 1 page poisoned)."""
    sb = 1 * 1000
    perm = _perm(4, sb + _T_PERM)
    ctx = [1, 200]
    return build_case("tiny-decode-b2-h8kv2", sb, ctx, 8, 2, 4, consecutive_runs(ctx, perm), 2,
                      device=device, with_new=with_new)


def qwen3_14b_decode_b16(device="cpu", with_new=False, pool_device=None) -> PagedCase:
    """Qwen3-14B decode step: batch 16, 40/8 heads, contexts uniform in [1, 4096],
    pages drawn from a shuffled 512-page pool."""
    sb = 2 * 1000
    ctx = torch.randint(1, 4097, (16,), generator=_gen(sb + _T_LEN)).tolist()
    perm = _perm(512, sb + _T_PERM)
    return build_case("qwen3-14b-decode-b16", sb, ctx, 40, 8, 512, consecutive_runs(ctx, perm), 32,
                      device=device, with_new=with_new, pool_device=pool_device)


def qwen3_14b_decode_b128(device="cpu", with_new=False, pool_device=None, poison=True,
                          batch=128) -> PagedCase:
    """Qwen3-14B bandwidth-bound decode: batch 128, every context 4096 (32 pages),
    block table a seeded permutation of the 4096-page pool (2.147 GB of K+V read).
    `batch` scales the batch and the pool together (32 pages per sequence)."""
    sb = 3 * 1000
    ctx = [4096] * batch
    perm = _perm(32 * batch, sb + _T_PERM)
    return build_case(f"qwen3-14b-decode-b{batch}-ctx4096", sb, ctx, 40, 8, 32 * batch,
                      consecutive_runs(ctx, perm), 32, device=device, with_new=with_new,
                      pool_device=pool_device, poison=poison)


def qwen3_32b_ragged(device="cpu", with_new=True, pool_device=None) -> PagedCase:
    """Qwen3-32B-shaped ragged decode: batch 64, 64/8 heads, contexts
    round(exp(U[ln 16, ln 4096])), a 3000-page pool of which a seeded 30% (900
    pages, interleaved) is free and NaN; the batch's pages are drawn in shuffled
    order from the 2100 allocated ones, the rest hold unrelated N(0,1) data.
    Includes the new token's KV write."""
    sb = 4 * 1000
    u = torch.rand(64, generator=_gen(sb + _T_LEN), dtype=torch.float64)
    ctx = [int(round(math.exp(math.log(16) + float(x) * (math.log(4096) - math.log(16))))) for x in u]
    perm = _perm(3000, sb + _T_PERM)
    free = set(perm[:900])
    allocated = [p for p in perm[900:]]  # already shuffled order
    need = sum((c + PAGE - 1) // PAGE for c in ctx)
    assert need <= len(allocated), need
    case = build_case("qwen3-32b-ragged-b64", sb, ctx, 64, 8, 3000,
                      consecutive_runs(ctx, allocated), 32, device=device, with_new=with_new,
                      poison=True, pool_device=pool_device)
    # Allocated pages outside the batch keep their N(0,1) data; only the free 30%
    # stays poisoned (build_case poisoned every unreferenced page).
    pdev = case.k_cache.device
    keep = sorted(set(case.poisoned_pages) - free)
    if keep:
        idx = torch.as_tensor(keep, dtype=torch.long, device=pdev)
        kf = randn_bf16((len(keep), PAGE, 8, HEAD_DIM), sb + 11, pdev)
        vf = randn_bf16((len(keep), PAGE, 8, HEAD_DIM), sb + 12, pdev)
        case.k_cache[idx] = kf
        case.v_cache[idx] = vf
    case.poisoned_pages = sorted(free)
    return case


def multi_token_decode(device="cpu", pool_device=None, B=64, q_len=4, ctx=4096, Hq=40, Hkv=8,
                       seed_index=6) -> PagedCase:
    """Multi-token decode (speculative-decoding verification): B sequences of
    context `ctx` after the write, the last q_len tokens new (K/V with the case,
    slots poisoned), 40/8 heads, a seeded permutation of a pool of exactly the
    pages used (64 x 4096 tokens: 1.07 GB of K+V)."""
    sb = seed_index * 1000
    ctxs = [ctx] * B
    need = B * ((ctx + PAGE - 1) // PAGE)
    perm = _perm(need, sb + _T_PERM)
    return build_case(f"multi-token-decode-b{B}-q{q_len}-ctx{ctx}", sb, ctxs, Hq, Hkv, need,
                      consecutive_runs(ctxs, perm), (ctx + PAGE - 1) // PAGE,
                      chunk_lens=[q_len] * B, with_new=True, device=device,
                      pool_device=pool_device)


def chunked_prefill(device="cpu", pool_device=None, B=8, chunk=512, Hq=40, Hkv=8,
                    max_prior=3584, seed_index=5) -> PagedCase:
    """Chunked paged prefill: 8 sequences packed token-major, 512 new tokens each
    (T = 4096), prior cached context uniform in [0, 3584], 40/8 heads.  The new
    tokens' K/V come with the case (the KV write precedes attention); their slots
    start poisoned."""
    sb = seed_index * 1000
    prior = torch.randint(0, max_prior + 1, (B,), generator=_gen(sb + _T_PRIOR)).tolist()
    ctx = [p + chunk for p in prior]
    maxp = (max_prior + chunk + PAGE - 1) // PAGE
    num_pages = B * maxp + 64
    perm = _perm(num_pages, sb + _T_PERM)
    return build_case(f"chunked-prefill-b{B}-c{chunk}", sb, ctx, Hq, Hkv, num_pages,
                      consecutive_runs(ctx, perm), maxp, chunk_lens=[chunk] * B,
                      with_new=True, device=device, pool_device=pool_device)


def custom_case(seed: int, ctx_lens, Hq=8, Hkv=2, chunk_lens=None, with_new=False,
                extra_pages: int = 3, max_pages_per_seq=None, device="cpu") -> PagedCase:
    """A small case with explicit lengths: a shuffled pool with `extra_pages`
    poisoned pages beyond what the sequences use."""
    need = [(c + PAGE - 1) // PAGE for c in ctx_lens]
    num_pages = max(1, sum(need) + extra_pages)
    perm = _perm(num_pages, seed + _T_PERM)
    mp = max_pages_per_seq or max(1, max(need) if need else 1)
    return build_case(f"custom-{seed}", seed, list(ctx_lens), Hq, Hkv, num_pages,
                      consecutive_runs(ctx_lens, perm), mp, chunk_lens=chunk_lens,
                      with_new=with_new, device=device)


CONFIGS = {
    "tiny": tiny_decode,
    "qwen3-14b-b16": qwen3_14b_decode_b16,
    "qwen3-14b-b128": qwen3_14b_decode_b128,
    "qwen3-32b-ragged": qwen3_32b_ragged,
    "chunked-prefill": chunked_prefill,
}


def prologue_inputs(case: PagedCase, seed: int, device="cpu"):
    """Inputs of the QK-norm / RoPE / KV-write prologue for `case`'s new tokens:
    the fused projection rows qkv [T, (Hq + 2 Hkv) * 128] bf16 ~ N(0, 1) and the
    FP32 per-head norm weights q_norm_w, k_norm_w [128] ~ U[0.5, 1.5]."""
    T = case.T
    row = (case.Hq + 2 * case.Hkv) * PAGE
    qkv = randn_bf16((T, row), seed + _T_QKV, device=device)
    wq = (torch.rand(PAGE, generator=_gen(seed + _T_WQ)) + 0.5).to(device)
    wk = (torch.rand(PAGE, generator=_gen(seed + _T_WK)) + 0.5).to(device)
    return qkv, wq, wk
