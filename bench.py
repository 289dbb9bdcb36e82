#!/usr/bin/env python
"""Benchmark of the paged-KV GQA attention hot path on one GB300.

Default workload: Qwen3-14B bandwidth-bound decode -- batch 128, every context
4096 tokens (32 pages of 128), 40 query heads over 8 KV heads, head_dim 128,
BF16 K/V ~ N(0,1) in a 4096-page pool under a seeded random block table.  One
step = pa_kv_write of each sequence's new token, then pa_decode (the
flash-decoding kernel plus its split combine).  The K+V read per step
(2.147 GB) is far larger than L2, so no flush is needed between steps.

Prints one JSON line (see the keys below).  `--impl reference` times the FP64
CPU oracle on a bounded sample of the same workload instead.
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged GQA decode attn: KV GB/s (% of GB300 HBM peak), seqs/s; prefill TFLOP/s"
UNIT = "GB/s"
WORKLOAD = "qwen3-14b-decode-b128-ctx4096"
B, HQ, HKV, D, PAGE, CTX = 128, 40, 8, 128, 128, 4096
KV_BYTES = B * CTX * HKV * D * 2 * 2          # K and V, bf16: 2.147 GB
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
PREFILL_WORKLOAD = "chunked-prefill-b8-c512"


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--num-splits", type=int, default=0,
                    help="0: automatic, -1: page-balanced, >= 1: fixed splits")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--batch", type=int, default=B,
                    help="decode batch (pool = 32 pages per sequence); smaller values are "
                         "for profiling captures, the benchmark workload is 128")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--profile-leg", choices=["prefill", "prefill-fp8", "fp8", "prologue", "topk", "multi",
                                              "decode-b16", "decode-ragged"],
                    default=None,
                    help="run one benchmark leg's calls a few times (FP8 and multi-token legs at "
                         "--batch sequences) for an ncu capture, then exit; prints no bench line")
    return ap.parse_args()


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        return float(m["hbm_gbs"]), float(m["bf16_tflops"]), float(m.get("bf16_tflops_sustained", m["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        import threading
        self.lines = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return self
        self.reader = threading.Thread(target=self._read, daemon=True)
        self.reader.start()
        # nvidia-smi takes a moment to start: wait (bounded) for its first line
        # so that short timed regions still get samples
        t0 = time.time()
        while not self.lines and time.time() - t0 < 5.0 and self.proc.poll() is None:
            time.sleep(0.01)
        self.skip = len(self.lines)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line)

    def __exit__(self, *a):
        self.out = ""
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.reader.join(timeout=5)
            # the samples taken before the timed region started are dropped
            # unless they are all there is
            got = self.lines[self.skip:] or self.lines
            self.out = "".join(got)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "samples": len(sm), "reasons": sorted(reasons)}


def dist_setup(args):
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if (args.impl == "ours" and torch.cuda.is_available()) else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available() and args.impl == "ours":
        torch.cuda.set_device(0)
    return ws, rank, local


def max_over_ranks(x, ws):
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def decode_traffic_from_profile():
    """dram bytes per decode launch from the committed ncu summary, if it was
    taken on the current decode kernel source (else None)."""
    import hashlib
    csrc = os.path.join(ROOT, "paged_kv_gqa_write_gb300", "csrc")
    prof = os.path.join(ROOT, "profiles", "decode_kernel_qwen3-14b-b16.md")
    try:
        # the decode path: its kernel, the combines and the shared device helpers
        blob = b"".join(open(os.path.join(csrc, f), "rb").read()
                        for f in ("pa_decode.cu", "pa_combine.cu", "pa_common.cuh"))
        h = hashlib.sha256(blob).hexdigest()[:16]
        vals = {}
        for line in open(prof):
            if ":" in line and line.strip().startswith("- "):
                k, v = line.strip()[2:].split(":", 1)
                # the value's first word (a hash in backquotes, or a number)
                vals[k.strip()] = v.strip().split()[0].strip("`") if v.strip() else ""
        if vals.get("source_sha256_16") != h:
            return None
        # captured on the batch-16 case; traffic scales with the units processed
        return float(vals["dram_bytes_per_launch"]) * B / 16.0
    except Exception:
        return None


def spread(ms_list):
    """Median, p10 and p90 (ms) of per-step event times."""
    v = sorted(ms_list)
    at = lambda q: v[min(len(v) - 1, int(q * (len(v) - 1) + 0.5))]
    return {"median_ms": statistics.median(v), "p10_ms": at(0.1), "p90_ms": at(0.9)}


def cpu_oracle_rate(case, seconds, rank0=True, threads=None):
    """Time the FP64 oracle on whole decode steps of `case` (host copies) until
    `seconds` have passed; returns (GB/s of K+V processed, threads, sample text).
    `threads`: OpenMP threads (default: all host cores)."""
    import oracle
    nt = threads or oracle.max_threads()
    kb = case.k_cache.cpu()
    vb = case.v_cache.cpu()
    q = case.q.cpu()
    bt = case.block_table.cpu()
    ctx = case.context_lens.cpu()
    rows_total = case.B * case.Hq
    # one chunk = 1/8 of a step (640 rows), so short budgets still finish
    import numpy as np
    chunk = max(1, rows_total // 8)
    done_rows, t0 = 0, time.perf_counter()
    i = 0
    while True:
        lo = (i * chunk) % rows_total
        rows = np.arange(lo, min(rows_total, lo + chunk), dtype=np.int64)
        oracle.attention(q, kb, vb, bt, ctx, None, case.scale, case.Hq, case.Hkv, case.num_pages,
                         case.max_pages_per_seq, rows=rows, num_threads=nt)
        done_rows += rows.shape[0]
        i += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    kv = KV_BYTES * done_rows / rows_total
    sample = (f"{done_rows} (sequence, query head) rows = {done_rows / rows_total:.2f} steps "
              f"of the {rows_total}-row workload, FP64, {nt} OpenMP threads, {el:.1f} s")
    return kv / el / 1e9, nt, sample


def run_reference(args):
    ws, rank, _ = dist_setup(args)
    if rank != 0:
        return
    import workloads as W
    from oracle import build as ob
    ob.build()
    case = W.qwen3_14b_decode_b128(device="cpu", with_new=False, poison=True)
    # each step: a bounded sample so that warmup + steps end within minutes
    per_step = max(1.0, min(10.0, 120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        cpu_oracle_rate(case, per_step / 4)
    vals, threads, sample = [], 0, ""
    for _ in range(args.steps):
        v, threads, sample = cpu_oracle_rate(case, per_step)
        vals.append(v)
    value = statistics.mean(vals)
    ms = KV_BYTES / (value * 1e9) * 1e3
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "batch": B, "context_len": CTX, "q_heads": HQ,
                       "kv_heads": HKV, "head_dim": D, "page_size": PAGE},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


class L2Flush:
    """Evicts L2 between timed steps: writes a buffer larger than L2, then
    reads another, so the timed kernel starts with clean (not dirty) lines."""

    def __init__(self, torch):
        self.w = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        self.r = torch.ones(64 << 20, dtype=torch.float32, device="cuda")

    def __call__(self):
        self.w.zero_()
        self.r.sum()


def run_decode_config(pa, W, torch, name, steps=50, warmup=10):
    """One of the smaller decode configurations, timed per step with an L2
    flush in between (their K+V is about the size of L2)."""
    if name == "qwen3-14b-decode-b16":
        case = W.qwen3_14b_decode_b16(device="cuda", pool_device="cuda")
        with_write = False
    else:
        case = W.qwen3_32b_ragged(device="cuda", pool_device="cuda")
        with_write = True
    kv_bytes = int(case.context_lens.sum()) * case.Hkv * D * 2 * 2
    out = torch.empty(case.B, case.Hq, D, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dims = pa.make_dims(case.B, case.Hq, case.Hkv, case.num_pages, case.max_pages_per_seq)
    sched = pa.pa_decode_auto_splits(dims)
    ws = torch.empty(max(1, pa.pa_decode_workspace_size(dims, 0)), dtype=torch.uint8,
                     device="cuda")

    def step():
        if with_write:
            pa.pa_kv_write(case.k_new, case.v_new, case.k_cache, case.v_cache,
                           case.block_table, case.context_lens, None, status=st)
        pa.pa_decode(case.q, case.k_cache, case.v_cache, case.block_table, case.context_lens,
                     case.scale, out=out, workspace=ws, num_splits=0, status=st)

    flush = L2Flush(torch)
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for a, b in ev:
        flush()
        a.record()
        step()
        b.record()
    torch.cuda.synchronize()
    sp = spread([a.elapsed_time(b) for a, b in ev])
    ms = sp["median_ms"]
    return {"workload": name, "batch": case.B, "q_heads": case.Hq, "kv_heads": case.Hkv,
            "spread": sp,
            "kv_bytes": kv_bytes, "ms": ms, "gbs": kv_bytes / (ms * 1e-3) / 1e9,
            "seqs_per_s": case.B / (ms * 1e-3), "status": int(st.item()),
            "schedule": "page-balanced" if sched == 0 else f"{sched} fixed splits",
            "step": ("pa_kv_write (1 token/seq) + " if with_write else "") + "pa_decode",
            "l2": "flushed between steps"}


def run_multi_token(pa, W, torch, hbm, steps=50, warmup=10, batch=64):
    """Multi-token decode (64 sequences x 4096 tokens, 4 new tokens each, 40/8
    heads): the 256 new tokens' KV write, then pa_decode_multi -- and the same
    attention through pa_prefill_chunk for comparison.  Bytes: the K+V of every
    context read once (1.07 GB; the working set is far larger than L2)."""
    q_len = 4
    case = W.multi_token_decode(device="cuda", pool_device="cuda", q_len=q_len, B=batch)
    kv_bytes = int(case.context_lens.sum()) * case.Hkv * D * 2 * 2
    out = torch.empty(case.T, case.Hq, D, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dims = pa.make_dims(case.B, case.Hq, case.Hkv, case.num_pages, case.max_pages_per_seq)
    ws = torch.empty(max(1, pa.pa_decode_multi_workspace_size(dims, q_len, 0)),
                     dtype=torch.uint8, device="cuda")
    sched = pa.pa_decode_auto_splits(pa.make_dims(case.B * q_len, case.Hq, case.Hkv,
                                                  case.num_pages, case.max_pages_per_seq))

    def write():
        pa.pa_kv_write(case.k_new, case.v_new, case.k_cache, case.v_cache, case.block_table,
                       case.context_lens, case.chunk_lens, status=st)

    def via_decode():
        write()
        pa.pa_decode_multi(case.q, case.k_cache, case.v_cache, case.block_table,
                           case.context_lens, q_len, case.scale, out=out, workspace=ws,
                           num_splits=0, status=st)

    def via_prefill():
        write()
        pa.pa_prefill_chunk(case.q, case.k_cache, case.v_cache, case.block_table,
                            case.context_lens, case.chunk_lens, case.scale, out=out, status=st)

    res = {"workload": f"multi-token-decode-b{case.B}-q{q_len}-ctx4096", "batch": case.B,
           "q_len": q_len, "q_heads": case.Hq, "kv_heads": case.Hkv, "kv_bytes": kv_bytes,
           "schedule": "page-balanced" if sched == 0 else f"{sched} fixed splits",
           "step": f"pa_kv_write ({case.T} tokens) + attention", "l2": "working set > L2"}
    for name, fn in (("pa_decode_multi", via_decode), ("pa_prefill_chunk", via_prefill)):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        for a, b in ev:
            a.record()
            fn()
            b.record()
        torch.cuda.synchronize()
        sp = spread([a.elapsed_time(b) for a, b in ev])
        ms = sp["median_ms"]
        gbs = kv_bytes / (ms * 1e-3) / 1e9
        res[name] = {"ms": ms, "spread": sp, "gbs": gbs, "frac": gbs / hbm,
                     "tokens_per_s": case.T / (ms * 1e-3)}
    res["status"] = int(st.item())
    return res


def run_fp8(pa, W, torch, hbm, steps=50, warmup=10, batch=128):
    """FP8 (e4m3) KV cache on the headline shape (128 sequences x 4096 tokens,
    40/8 heads): the new token's quantizing write, then pa_decode_fp8 over
    1.07 GB of e4m3 K+V (the working set is far larger than L2)."""
    case = W.qwen3_14b_decode_b128(device="cuda", pool_device="cuda", with_new=True,
                                   poison=False, batch=batch)
    Hkv = case.Hkv
    g = torch.Generator(device="cuda").manual_seed(11)
    ks = torch.rand(Hkv, generator=g, device="cuda") * 0.02 + 0.02
    vs = torch.rand(Hkv, generator=g, device="cuda") * 0.02 + 0.02
    k8 = (case.k_cache.float() / ks[None, None, :, None]).to(torch.float8_e4m3fn).view(torch.uint8)
    v8 = (case.v_cache.float() / vs[None, None, :, None]).to(torch.float8_e4m3fn).view(torch.uint8)
    del case.k_cache, case.v_cache
    kv_bytes = int(case.context_lens.sum()) * Hkv * D * 2   # e4m3 K + V
    out = torch.empty(case.B, case.Hq, D, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dims = pa.make_dims(case.B, case.Hq, Hkv, k8.shape[0], case.max_pages_per_seq)
    ws = torch.empty(max(1, pa.pa_decode_multi_workspace_size(dims, 1, 0)), dtype=torch.uint8,
                     device="cuda")

    def step():
        pa.pa_kv_write_fp8(case.k_new, case.v_new, k8, v8, ks, vs, case.block_table,
                           case.context_lens, None, status=st)
        pa.pa_decode_fp8(case.q, k8, v8, ks, vs, case.block_table, case.context_lens, 1,
                         case.scale, out=out, workspace=ws, num_splits=0, status=st)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for a, b in ev:
        a.record()
        step()
        b.record()
    torch.cuda.synchronize()
    sp = spread([a.elapsed_time(b) for a, b in ev])
    ms = sp["median_ms"]
    gbs = kv_bytes / (ms * 1e-3) / 1e9
    return {"workload": f"qwen3-14b-decode-b{batch}-ctx4096-fp8-kv", "kv_bytes": kv_bytes, "ms": ms,
            "spread": sp,
            "gbs": gbs, "frac": gbs / hbm, "bf16_equivalent_gbs": 2 * gbs,
            "status": int(st.item()), "step": "pa_kv_write_fp8 (1 token/seq) + pa_decode_fp8",
            "l2": "working set > L2"}


def run_prologue(pa, W, torch, hbm, steps=50, warmup=10):
    """pa_qk_norm_rope_write (Q/K RMSNorm -> NeoX RoPE -> KV write) on the decode
    batch (128 tokens), on the 8 x 512 prefill chunk and on the batch-16 decode,
    with a clean L2 flush between steps.  Bytes: the fused QKV rows read, Q and
    the K/V rows written.  For the decode batches also the decode step behind
    it: pa_decode alone, the prologue then pa_decode, and pa_decode_prologue."""
    out = {}
    flush = L2Flush(torch)
    for name, case in (("decode-b128", W.qwen3_14b_decode_b128(device="cuda", pool_device="cuda",
                                                                with_new=False)),
                       ("prefill-b8-c512", W.chunked_prefill(device="cuda", pool_device="cuda")),
                       ("decode-b16", W.qwen3_14b_decode_b16(device="cuda", pool_device="cuda"))):
        qkv, wq, wk = W.prologue_inputs(case, 600, device="cuda")
        chunked = case.chunk_lens is not None
        q_out = torch.empty(case.T, case.Hq, D, dtype=torch.bfloat16, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")

        def step():
            pa.pa_qk_norm_rope_write(qkv, wq, wk, case.k_cache, case.v_cache, case.block_table,
                                     case.context_lens, case.chunk_lens if chunked else None,
                                     q_scale=1.0 / math.sqrt(D), q_out=q_out, status=st)

        for _ in range(warmup):
            step()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        for a, b in ev:
            flush()
            a.record()
            step()
            b.record()
        torch.cuda.synchronize()
        sp = spread([a.elapsed_time(b) for a, b in ev])
        ms = sp["median_ms"]
        nbytes = case.T * (case.Hq + 2 * case.Hkv) * D * 2 * 2
        out[name] = {"tokens": case.T, "us": ms * 1e3, "spread": sp, "bytes": nbytes,
                     "gbs": nbytes / (ms * 1e-3) / 1e9, "frac": nbytes / (ms * 1e-3) / 1e9 / hbm,
                     "status": int(st.item())}
        # the same prologue into an FP8 (e4m3) cache: K/V rows stored as codes
        ks = torch.full((case.Hkv,), 0.03, dtype=torch.float32, device="cuda")
        k8 = torch.zeros(case.k_cache.shape, dtype=torch.uint8, device="cuda")
        v8 = torch.zeros_like(k8)

        def step8():
            pa.pa_qk_norm_rope_write_fp8(qkv, wq, wk, k8, v8, ks, ks, case.block_table,
                                         case.context_lens, case.chunk_lens if chunked else None,
                                         q_scale=1.0 / math.sqrt(D), q_out=q_out, status=st)

        for _ in range(warmup):
            step8()
        torch.cuda.synchronize()
        ev8 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        for a, b in ev8:
            flush()
            a.record()
            step8()
            b.record()
        torch.cuda.synchronize()
        sp8 = spread([a.elapsed_time(b) for a, b in ev8])
        b8 = case.T * D * ((case.Hq + 2 * case.Hkv) * 2 + case.Hq * 2 + 2 * case.Hkv)
        out[name]["fp8_cache"] = {"step": "pa_qk_norm_rope_write_fp8", "us": sp8["median_ms"] * 1e3,
                                  "spread": sp8, "bytes": b8,
                                  "gbs": b8 / (sp8["median_ms"] * 1e-3) / 1e9,
                                  "frac": b8 / (sp8["median_ms"] * 1e-3) / 1e9 / hbm,
                                  "status": int(st.item())}
        del k8, v8
        if not chunked:
            # the decode step behind the prologue: pa_decode alone, and the
            # prologue (128 tokens) then pa_decode, each timed the same way
            dims = pa.make_dims(case.B, case.Hq, case.Hkv, case.num_pages, case.max_pages_per_seq)
            wsp = torch.empty(max(1, pa.pa_decode_workspace_size(dims, 0)), dtype=torch.uint8,
                              device="cuda")
            dout = torch.empty(case.B, case.Hq, D, dtype=torch.bfloat16, device="cuda")

            def dec():
                pa.pa_decode(q_out, case.k_cache, case.v_cache, case.block_table,
                             case.context_lens, 1.0, out=dout, workspace=wsp, num_splits=0,
                             status=st)

            def chain():
                step()
                dec()

            def fused():
                pa.pa_decode_prologue(qkv, wq, wk, case.k_cache, case.v_cache, case.block_table,
                                      case.context_lens, q_scale=1.0 / math.sqrt(D), scale=1.0,
                                      out=dout, workspace=wsp, num_splits=0, status=st)

            res = {}
            for leg, fn in (("pa_decode", dec), ("pa_qk_norm_rope_write + pa_decode", chain),
                            ("pa_decode_prologue", fused)):
                for _ in range(warmup):
                    fn()
                torch.cuda.synchronize()
                evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                       for _ in range(steps)]
                for a, b in evs:
                    flush()
                    a.record()
                    fn()
                    b.record()
                torch.cuda.synchronize()
                res[leg] = spread([a.elapsed_time(b) for a, b in evs])["median_ms"] * 1e3
            out[name]["decode_step_us"] = res
            out[name]["prologue_cost_in_step_us"] = res["pa_qk_norm_rope_write + pa_decode"] - res["pa_decode"]
            out[name]["fused_prologue_cost_in_step_us"] = res["pa_decode_prologue"] - res["pa_decode"]
    out["step"] = "pa_qk_norm_rope_write"
    out["l2"] = "flushed between steps"
    return out


def run_topk(pa, torch, hbm, steps=50, warmup=10):
    """Exact top-32 of 16 rows of 151936 logits (the Qwen3-14B real vocabulary in
    rows padded to 152064), the selector's batch-16 configuration; L2 flushed
    between steps.  Bytes: the logits read once."""
    g = torch.Generator(device="cuda").manual_seed(706)
    buf = torch.randn(16, 152064, generator=g, device="cuda", dtype=torch.float32)
    logits = buf[:, :151936]
    vals = torch.empty(16, 32, dtype=torch.float32, device="cuda")
    idx = torch.empty(16, 32, dtype=torch.int32, device="cuda")
    ws = torch.empty(max(16, pa.load().pa_topk_workspace_size(16, 151936, 32)), dtype=torch.uint8,
                     device="cuda")
    flush = L2Flush(torch)

    def step():
        pa.pa_topk(logits, 32, out_values=vals, out_indices=idx, workspace=ws)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for a, b in ev:
        flush()
        a.record()
        step()
        b.record()
    torch.cuda.synchronize()
    sp = spread([a.elapsed_time(b) for a, b in ev])
    ms = sp["median_ms"]
    nbytes = 16 * 151936 * 4
    ref = torch.topk(logits, 32, dim=1)
    exact = bool(torch.equal(ref.indices.to(torch.int32), idx)) and bool(torch.equal(ref.values, vals))
    return {"workload": "topk-b16-v151936-k32", "us": ms * 1e3, "spread": sp, "bytes": nbytes,
            "gbs": nbytes / (ms * 1e-3) / 1e9, "frac": nbytes / (ms * 1e-3) / 1e9 / hbm,
            "matches_torch_topk": exact, "step": "pa_topk (slice select + merge)",
            "l2": "flushed between steps"}


def run_prefill(pa, W, torch, steps=50, warmup=10, fp8=False):
    """Chunked prefill (8 x 512 new tokens): KV write then causal attention.
    fp8: the same over an FP8 (e4m3) cache with per-KV-head scales
    (pa_kv_write_fp8 + pa_prefill_chunk_fp8)."""
    case = W.chunked_prefill(device="cuda", pool_device="cuda")
    flops = 0.0
    for s in range(case.B):
        n = int(case.chunk_lens[s])
        prior = int(case.context_lens[s]) - n
        flops += case.Hq * 4 * D * sum(prior + j + 1 for j in range(n))
    out = torch.empty(case.T, case.Hq, D, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    if fp8:
        g = torch.Generator(device="cuda").manual_seed(13)
        ks = torch.rand(case.Hkv, generator=g, device="cuda") * 0.02 + 0.02
        vs = torch.rand(case.Hkv, generator=g, device="cuda") * 0.02 + 0.02
        k8 = (case.k_cache.float() / ks[None, None, :, None]).to(torch.float8_e4m3fn).view(torch.uint8)
        v8 = (case.v_cache.float() / vs[None, None, :, None]).to(torch.float8_e4m3fn).view(torch.uint8)
        del case.k_cache, case.v_cache

        def step():
            pa.pa_kv_write_fp8(case.k_new, case.v_new, k8, v8, ks, vs, case.block_table,
                               case.context_lens, case.chunk_lens, status=st)
            pa.pa_prefill_chunk_fp8(case.q, k8, v8, ks, vs, case.block_table, case.context_lens,
                                    case.chunk_lens, case.scale, out=out, status=st)
    else:
        def step():
            pa.pa_kv_write(case.k_new, case.v_new, case.k_cache, case.v_cache, case.block_table,
                           case.context_lens, case.chunk_lens, status=st)
            pa.pa_prefill_chunk(case.q, case.k_cache, case.v_cache, case.block_table,
                                case.context_lens, case.chunk_lens, case.scale, out=out, status=st)

    flush = L2Flush(torch)
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for a, b in ev:
        flush()                            # L2 flush between steps (working set < L2)
        a.record()
        step()
        b.record()
    torch.cuda.synchronize()
    sp = spread([a.elapsed_time(b) for a, b in ev])
    ms = sp["median_ms"]
    name = "pa_kv_write_fp8 (4096 tokens) + pa_prefill_chunk_fp8" if fp8 else \
        "pa_kv_write (4096 tokens) + pa_prefill_chunk"
    return {"workload": PREFILL_WORKLOAD + ("-fp8-kv" if fp8 else ""),
            "tflops": flops / (ms * 1e-3) / 1e12, "ms": ms, "spread": sp,
            "gflop_causal": flops / 1e9, "status": int(st.item()),
            "step": name, "l2": "flushed between steps"}


def run_ours(args):
    global B, KV_BYTES, WORKLOAD
    if args.batch != B:
        B = args.batch
        KV_BYTES = B * CTX * HKV * D * 2 * 2
        WORKLOAD = f"qwen3-14b-decode-b{B}-ctx4096"
    import torch
    ws, rank, local = dist_setup(args)
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_gqa_write_gb300 as pa
    import workloads as W

    if args.profile_leg:
        hbm_p = peaks()[0]
        if args.profile_leg == "prefill":
            r = run_prefill(pa, W, torch, steps=2, warmup=1)
        elif args.profile_leg == "prefill-fp8":
            r = run_prefill(pa, W, torch, steps=2, warmup=1, fp8=True)
        elif args.profile_leg == "fp8":
            r = run_fp8(pa, W, torch, hbm_p, steps=2, warmup=1, batch=args.batch)
        elif args.profile_leg == "prologue":
            r = run_prologue(pa, W, torch, hbm_p, steps=2, warmup=1)
        elif args.profile_leg == "topk":
            r = run_topk(pa, torch, hbm_p, steps=2, warmup=1)
        elif args.profile_leg == "decode-b16":
            r = run_decode_config(pa, W, torch, "qwen3-14b-decode-b16", steps=2, warmup=1)
        elif args.profile_leg == "decode-ragged":
            r = run_decode_config(pa, W, torch, "qwen3-32b-ragged-b64", steps=2, warmup=1)
        else:
            r = run_multi_token(pa, W, torch, hbm_p, steps=2, warmup=1, batch=args.batch)
        print(json.dumps({"profile_leg": args.profile_leg, "batch": args.batch,
                          "status": r.get("status", 0)}), flush=True)
        return

    dev = torch.device("cuda", torch.cuda.current_device())
    case = W.qwen3_14b_decode_b128(device=dev, with_new=True, pool_device=dev, batch=B)
    dims = pa.make_dims(B, HQ, HKV, case.num_pages, case.max_pages_per_seq)
    # schedule: fixed split count >= 1, or 0 / PA_SPLITS_BALANCED for page-balanced
    splits = args.num_splits if args.num_splits != 0 else pa.pa_decode_auto_splits(dims)
    balanced = splits in (0, pa.PA_SPLITS_BALANCED)
    if balanced:
        splits = pa.PA_SPLITS_BALANCED
    ws_bytes = pa.pa_decode_workspace_size(dims, splits)
    workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    out = torch.empty(B, HQ, D, dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    def step(ev=None):
        pa.pa_kv_write(case.k_new, case.v_new, case.k_cache, case.v_cache, case.block_table,
                       case.context_lens, None, status=status, stream=stream)
        if ev is not None:
            ev[0].record(stream)
        pa.pa_decode(case.q, case.k_cache, case.v_cache, case.block_table, case.context_lens,
                     case.scale, out=out, workspace=workspace, num_splits=splits, status=status,
                     stream=stream)
        if ev is not None:
            ev[1].record(stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"

    dec_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        start.record(stream)
        for i in range(args.steps):
            step(dec_ev[i])
        end.record(stream)
        torch.cuda.synchronize()
        barrier(ws)
    elapsed_ms = max_over_ranks(start.elapsed_time(end), ws)
    ms_per_step = elapsed_ms / args.steps
    dec_ms = statistics.mean(a.elapsed_time(b) for a, b in dec_ev)
    # a timed region of a few ms holds one or two samples at the sampler's
    # 100 ms period: a second record spans every later leg (seconds of load)
    clk_legs = ClockSampler(local).__enter__()
    # kv_write + decode, + a combine for the balanced schedule or fixed splits > 1
    launches_per_step = 2 + (1 if (balanced or splits > 1) else 0)

    # ---- end to end through the C ABI with host buffers (pinned), copies timed.
    # A step's inputs (q, the new K/V rows, the block table, the lengths) sit in
    # one pinned staging buffer and go up in one copy; the output comes back.
    # Pipelined (the value reported as e2e): two device staging slots and two
    # outputs, step k + 1's upload on one copy stream and step k's download on
    # another, both overlapping the kernels; events keep a slot from being
    # overwritten before its kernels (or its download) are done.  Serial: the
    # same copies and kernels in order on one stream.
    parts = (case.q, case.k_new, case.v_new, case.block_table, case.context_lens)
    offs, total = [], 0
    for t in parts:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    hstage = torch.empty(total, dtype=torch.uint8).pin_memory()
    for t, o in zip(parts, offs):
        n = t.numel() * t.element_size()
        hstage[o:o + n].copy_(t.cpu().contiguous().view(-1).view(torch.uint8))
    dstage = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(2)]
    views = []
    for b in range(2):
        vs = []
        for t, o in zip(parts, offs):
            n = t.numel() * t.element_size()
            vs.append(dstage[b][o:o + n].view(t.dtype).view(t.shape))
        views.append(vs)
    outs = [out, torch.empty_like(out)]
    houts = [torch.empty(B, HQ, D, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    h2d = total
    d2h = houts[0].numel() * houts[0].element_size()
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "used", "down")}

    def kernels(b):
        dq, dk, dv, dbt, dctx = views[b]
        pa.pa_kv_write(dk, dv, case.k_cache, case.v_cache, dbt, dctx, None, status=status,
                       stream=stream)
        pa.pa_decode(dq, case.k_cache, case.v_cache, dbt, dctx, case.scale, out=outs[b],
                     workspace=workspace, num_splits=splits, status=status, stream=stream)

    def e2e_serial_step():
        dstage[0].copy_(hstage, non_blocking=True)
        kernels(0)
        houts[0].copy_(outs[0], non_blocking=True)

    def e2e_pipelined(nsteps, start_ev):
        up.wait_event(start_ev)
        for k in range(nsteps):
            b = k & 1
            with torch.cuda.stream(up):
                if k >= 2:
                    up.wait_event(ev["used"][b])       # step k - 2's kernels read slot b
                dstage[b].copy_(hstage, non_blocking=True)
                ev["in"][b].record(up)
            stream.wait_event(ev["in"][b])
            if k >= 2:
                stream.wait_event(ev["down"][b])       # step k - 2's output went down
            kernels(b)
            ev["used"][b].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(ev["used"][b])
                houts[b].copy_(outs[b], non_blocking=True)
                ev["down"][b].record(down)
        for b in range(min(2, nsteps)):
            stream.wait_event(ev["down"][b])

    e2e_ms = e2e_serial_ms = None
    if not args.no_e2e:
        e2e_steps = max(10, args.steps // 4)
        for _ in range(3):
            e2e_serial_step()
        torch.cuda.synchronize()
        s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(ws)
        s2.record(stream)
        for _ in range(e2e_steps):
            e2e_serial_step()
        e2.record(stream)
        torch.cuda.synchronize()
        e2e_serial_ms = max_over_ranks(s2.elapsed_time(e2), ws) / e2e_steps
        w0 = torch.cuda.Event()
        w0.record(stream)
        e2e_pipelined(3, w0)
        torch.cuda.synchronize()
        s3, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(ws)
        s3.record(stream)
        e2e_pipelined(e2e_steps, s3)
        e3.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(s3.elapsed_time(e3), ws) / e2e_steps
    assert int(status.item()) == 0, f"device status {int(status.item())}"

    hbm, bf16, bf16_sus, src = peaks()
    value = KV_BYTES * ws / (ms_per_step * 1e-3) / 1e9
    achieved = KV_BYTES / (dec_ms * 1e-3) / 1e9
    prefill = None
    if not args.no_prefill:
        try:
            prefill = run_prefill(pa, W, torch)
            prefill["peak_tflops"] = bf16
            prefill["frac"] = prefill["tflops"] / bf16
        except Exception as e:  # report, do not hide
            prefill = {"error": str(e).splitlines()[0][:200]}
    prefill_fp8 = None
    if not args.no_prefill:
        try:
            prefill_fp8 = run_prefill(pa, W, torch, fp8=True)
            prefill_fp8["peak_tflops"] = bf16
            prefill_fp8["frac"] = prefill_fp8["tflops"] / bf16
            prefill_fp8["peak_note"] = "F16 products: the F16 dense rate equals BF16's"
        except Exception as e:  # report, do not hide
            prefill_fp8 = {"error": str(e).splitlines()[0][:200]}
    prologue = None
    if not args.no_prefill:
        try:
            prologue = run_prologue(pa, W, torch, hbm)
        except Exception as e:  # report, do not hide
            prologue = {"error": str(e).splitlines()[0][:200]}
    fp8 = None
    if not args.no_prefill:
        try:
            fp8 = run_fp8(pa, W, torch, hbm)
        except Exception as e:  # report, do not hide
            fp8 = {"error": str(e).splitlines()[0][:200]}
    multi = None
    if not args.no_prefill:
        try:
            multi = run_multi_token(pa, W, torch, hbm)
        except Exception as e:  # report, do not hide
            multi = {"error": str(e).splitlines()[0][:200]}
    topk = None
    if not args.no_prefill:
        try:
            topk = run_topk(pa, torch, hbm)
        except Exception as e:  # report, do not hide
            topk = {"error": str(e).splitlines()[0][:200]}
    other = None
    if not args.no_prefill:
        other = []
        for name in ("qwen3-14b-decode-b16", "qwen3-32b-ragged-b64"):
            try:
                r = run_decode_config(pa, W, torch, name)
                r["frac"] = r["gbs"] / hbm
                other.append(r)
            except Exception as e:  # report, do not hide
                other.append({"workload": name, "error": str(e).splitlines()[0][:200]})
    clk_legs.__exit__(None, None, None)  # (the GPU idles during the CPU baseline)
    clocks_legs = clk_legs.summary()
    clocks_legs["span"] = "the e2e runs and every GPU leg after the headline's timed region"
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        v, nt, sample = cpu_oracle_rate(case, args.cpu_seconds)
        v1, _, sample1 = cpu_oracle_rate(case, max(1.0, args.cpu_seconds / 4), threads=1)
        cpu = {"value": v, "unit": UNIT, "cores": nt, "kind": "oracle", "sample": sample,
               "single_thread": {"value": v1, "unit": UNIT, "sample": sample1}}
    clocks = clk.summary()
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "accum_dtype": "f32",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "batch": B, "context_len": CTX, "q_heads": HQ,
                   "kv_heads": HKV, "head_dim": D, "page_size": PAGE,
                   "kv_bytes_per_step": KV_BYTES,
                   "schedule": "page-balanced" if balanced else f"{splits} fixed splits",
                   "step": "pa_kv_write (1 token/seq) + pa_decode (decode kernel + combine)",
                   "l2": f"inputs larger than L2 ({KV_BYTES / 1e9:.3f} GB K+V per step), no flush",
                   "parallelism": f"replicas{ws}" if ws > 1 else "single-gpu"},
        "seqs_per_s": B * ws / (ms_per_step * 1e-3),
        "pct_hbm_peak": 100.0 * value / ws / hbm,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "traffic": decode_traffic_from_profile(),
                     "kernel": "pa_decode (decode_kernel + combine_kernel)",
                     "peak_source": f"{src} hbm_gbs (burst)",
                     "ms_per_launch": dec_ms,
                     "launch_spread": spread([a.elapsed_time(b) for a, b in dec_ev])},
        "e2e": None if e2e_ms is None else {
            "value": KV_BYTES * ws / (e2e_serial_ms * 1e-3) / 1e9, "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_serial_ms,
            "copies": "upload, kernels, download in order on one stream, every step",
            "pipelined": {"value": KV_BYTES * ws / (e2e_ms * 1e-3) / 1e9, "ms_per_step": e2e_ms,
                          "copies": "the same copies, double-buffered on two copy streams "
                                    "overlapping the previous and next steps' kernels"}},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "clocks_legs": clocks_legs,
        "prefill": prefill,
        "prefill_fp8_kv": prefill_fp8,
        "decode_configs": other,
        "prologue": prologue,
        "topk": topk,
        "multi_token_decode": multi,
        "fp8_kv_decode": fp8,
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
