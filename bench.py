#!/usr/bin/env python3
"""Benchmark of one decode step over an FP8-quantised, paged KV cache.

A step is the whole hot path for one batch: append every request's new
token (absmax scale, FP8 rounding, slot scatter) and run paged decode
attention over the full cache (plan, split kernel, merge).  The default
workload is one Llama-3-70B-shaped decode layer: 12 requests x 16384 cached
tokens, 64 query / 8 KV heads, head_dim 128, E4M3 codes with one scale per
(token, kv head), block size 16 -- 415 MB of cache read per step, more than
the 129 MB L2, so no flush is needed between steps.

Output: one JSON line (rank 0).  `value` is the achieved algorithmic HBM
bandwidth of the step in GB/s; `roofline` is for the split kernel alone,
timed with CUDA events around its launch; `append_roofline` is the bulk
(prefill) append of one request; `per_workload` repeats the split-kernel
measurement on the other full-size workloads (long context, ragged E5M2,
MLA latent); `e2e` is the same metric through the public API with pinned
host inputs copied in and the output copied back inside the timed region
(a replayed CUDA graph; `e2e_plain_call` the same with plain calls);
`cpu_baseline` times the CPU oracle on a bounded sample of the same
workload.  Working sets under 2 x L2 are flushed from L2 before every
timed step.

Multi-GPU (torchrun): replicas only -- every rank runs its own copy of the
workload with no collective on the data path (weak scaling); the step time
is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from fp8_quantised_paged_gb300 import workloads as W  # noqa: E402

METRIC = "FP8 paged decode attn: achieved HBM GB/s (% of GB300 peak), KV tokens/s"


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["fp8pa", "reference"], default="fp8pa")
    ap.add_argument("--workload", type=int, default=2, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--mx-block", type=int, default=0, choices=[0, 16, 32],
                    help="store the GQA workload's cache in the MX block-scaled mode "
                         "(one E8M0 exponent per block of this many dims)")
    ap.add_argument("--scale-mode", choices=["segment"], default=None,
                    help="store the GQA/MLA workload's cache with block-wise cumulative "
                         "rescaling: one scale per (page, KV head), refreshed every 1024 tokens")
    ap.add_argument("--kv-fmt", choices=["e4m3", "e5m2", "int8"], default=None,
                    help="store the workload's cache in this code format instead of its own")
    ap.add_argument("--q-len", type=int, default=1,
                    help="queries per request: a causal chunk (the last q_len tokens of each "
                         "request are appended, then attend); 1 is plain decode")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-per-workload", action="store_true",
                    help="skip the split-kernel lines of the other full-size workloads")
    ap.add_argument("--no-append-roofline", action="store_true",
                    help="skip the bulk (prefill) append measurement")
    ap.add_argument("--traffic-json", default=os.path.join(ROOT, "profiles", "traffic.json"),
                    help="per-launch DRAM bytes of the split kernel from an ncu capture")
    return ap.parse_args()


# ---------------------------------------------------------------- accounting
def accounting(w: W.Workload, b_sel=None, q_len: int = 1) -> dict:
    """Algorithmic bytes of one step (or of the requests in b_sel): the cache
    is read once however many queries a request has in its chunk."""
    bs = w.block_size
    lens = w.seq_lens if b_sel is None else w.seq_lens[list(b_sel)]
    B = len(lens)
    ntens = 1 if w.mla else 2
    kv_tokens = int(lens.sum())
    codes = w.head_dim * w.n_kv_heads * ntens
    if w.scale_mode == W.SCALE_TOKEN_HEAD:
        sc_tok = 4 * w.n_kv_heads * ntens
    elif w.scale_mode == W.SCALE_TOKEN_GROUP:
        sc_tok = 4 * w.n_kv_heads * (w.head_dim // w.group_size) * ntens
    elif w.scale_mode == W.SCALE_MX_BLOCK:  # one E8M0 byte per block
        sc_tok = w.n_kv_heads * (w.head_dim // w.group_size) * ntens
    else:
        sc_tok = 0
    static_sc = (4 * w.n_kv_heads * w.head_dim * ntens
                 if w.scale_mode == W.SCALE_CHANNEL_STATIC else 0)
    pages = int(sum(math.ceil(int(L) / bs) for L in lens))
    # segment mode: one f32 per (page, KV head) per tensor
    seg_sc = 4 * w.n_kv_heads * ntens * pages if w.scale_mode == W.SCALE_SEGMENT else 0
    kv = kv_tokens * (codes + sc_tok) + static_sc + seg_sc
    q = B * q_len * w.n_q_heads * w.head_dim * 2
    out = B * q_len * w.n_q_heads * w.head_dim_v * 2
    tables = pages * 4 + B * 4
    split = kv + q + tables
    decode = split + out
    append = B * q_len * (codes * 2 + codes + sc_tok + 4)
    if w.scale_mode == W.SCALE_SEGMENT:  # page-scale writes, state read and written
        append += B * q_len * 4 * w.n_kv_heads * ntens + B * 2 * (2 * w.n_kv_heads * 2 * 4)
    return {"kv_tokens": kv_tokens, "bytes_per_token": codes + sc_tok, "split": split,
            "decode": decode, "append": append, "step": decode + append}


def bench_workload(args) -> W.Workload:
    """The named full-size workload, optionally with an MX block-scaled cache
    or another code format."""
    w = W.make_workload(args.workload, "full")
    if args.kv_fmt is not None:
        fmt = {"e4m3": W.E4M3, "e5m2": W.E5M2, "int8": W.INT8}[args.kv_fmt]
        if fmt != w.fmt:
            w.fmt = fmt
            w.name = f"{w.name}_{args.kv_fmt}"
    if args.scale_mode == "segment":
        if args.mx_block:
            raise SystemExit("--scale-mode segment and --mx-block are exclusive")
        w.scale_mode, w.group_size = W.SCALE_SEGMENT, w.head_dim
        w.name = f"{w.name}_segment"
    if args.mx_block:
        if w.fmt == W.INT8:
            raise SystemExit("--mx-block needs FP8 codes")
        if w.mla:
            raise SystemExit("--mx-block applies to the grouped-query workloads")
        w.scale_mode, w.group_size = W.SCALE_MX_BLOCK, args.mx_block
        w.name = f"{w.name}_mx{args.mx_block}"
    return w


def scale_groups(w) -> int:
    grouped = (W.SCALE_TOKEN_GROUP, W.SCALE_MX_BLOCK)
    return w.head_dim // w.group_size if w.scale_mode in grouped else 1


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        # raw samples: FP8PA_CLOCKS_DIR if set (to keep them), else a temp dir
        out_dir = os.environ.get("FP8PA_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(out_dir, f"fp8pa_clocks_rank{index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index),
                                          f"--query-gpu={self.FIELDS}", "--format=csv,noheader",
                                          "-lms", "50"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sms, maxs, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1].split()[0]))
                maxs.append(float(parts[2].split()[0]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sms:
            return None
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxs),
                "reasons": sorted(reasons), "samples": len(sms)}


# ---------------------------------------------------------------- helpers
def peaks() -> dict:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


def flops_per_step(w: W.Workload) -> int:
    """Algorithmic attention flops: 2 x (QK^T + PV) multiply-adds."""
    return 2 * int(w.seq_lens.sum()) * w.n_q_heads * (w.head_dim + w.head_dim_v)


def kernel_source_sha(name="decode_gqa.cu") -> str:
    import hashlib
    with open(os.path.join(ROOT, "fp8_quantised_paged_gb300", "csrc", name), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def traffic_per_launch(path, workload_name, source="decode_gqa.cu"):
    """DRAM bytes per launch of the split kernel from the recorded ncu
    capture, or None when none was recorded for this workload or the
    kernel source changed since."""
    try:
        with open(path) as f:
            d = json.load(f)
        e = d.get(workload_name)
        if e is None or e.get("kernel_source_sha256") != kernel_source_sha(source):
            return None
        return float(e["dram_bytes_per_launch"])
    except (OSError, ValueError, KeyError, TypeError):
        return None


def max_over_ranks(x: float, device) -> float:
    """The maximum of a per-rank time over all ranks (the job's time)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def to_bf16_tensor(bits, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


# ---------------------------------------------------------------- CPU oracle timing
def oracle_sample(w: W.Workload, b: int, heads=None, threads=None):
    """Run the oracle (append of request b's tokens into a compact pool, then
    attention for `heads` of request b).  Returns (seconds, bytes)."""
    import oracle
    k, v = W.request_kv(w, b)
    L = int(w.seq_lens[b])
    bs, hkv, d = w.block_size, w.n_kv_heads, w.head_dim
    nbl = (L + bs - 1) // bs
    ng = scale_groups(w)
    kc = np.zeros((nbl, hkv, bs, d), np.uint8)
    vc = None if w.mla else np.zeros_like(kc)
    if w.scale_mode == W.SCALE_CHANNEL_STATIC:
        ks = oracle.kv_channel_scales(k, w.fmt)
        vs = oracle.kv_channel_scales(v, w.fmt)
    elif w.scale_mode == W.SCALE_SEGMENT:
        ks = np.zeros((nbl, oracle.segment_scale_heads(hkv)), np.float32)
        vs = None if w.mla else np.zeros_like(ks)
    else:
        ks = np.zeros((nbl, hkv, bs, ng),
                      np.uint8 if w.scale_mode == W.SCALE_MX_BLOCK else np.float32)
        vs = None if w.mla else np.zeros_like(ks)
    t = np.arange(L)
    slots = (t // bs * bs + t % bs).astype(np.int32)
    bt = np.arange(nbl, dtype=np.int32)[None]
    sl = np.array([L], np.int32)
    q = W.queries(w)[b:b + 1]
    heads = list(range(w.n_q_heads)) if heads is None else list(heads)
    t0 = time.perf_counter()
    if w.scale_mode == W.SCALE_SEGMENT:
        st = np.zeros((1, 2, hkv, 2), np.float32)
        oracle.kv_append_quant_segment(k, v, slots, [0, L], [0], w.fmt, st, kc, vc, ks, vs, bs)
    else:
        oracle.kv_append_quant(k, v, slots, w.fmt, w.scale_mode, w.group_size, kc, vc, ks, vs,
                               bs)
    if w.mla:
        vc, vs = kc, ks
    oracle.paged_decode_attention(q, kc, vc, ks, vs, bt, sl, bs, hkv, w.head_dim_v, w.fmt,
                                  w.scale_mode, w.group_size, w.sm_scale,
                                  rows=np.array(heads, np.int32), num_threads=threads)
    dt = time.perf_counter() - t0
    acc = accounting(w, [b])
    frac = len(heads) / w.n_q_heads
    return dt, acc["step"] * frac, acc["kv_tokens"] * frac


def run_reference(args, rank):
    """The CPU oracle as the reference arm: every step is a bounded sample
    (one request, one KV head's query group) of the same workload."""
    import oracle
    if rank != 0:
        return
    w = bench_workload(args)
    G = w.n_q_heads // w.n_kv_heads
    threads = oracle.max_threads()
    times, nbytes, toks = [], 0.0, 0.0
    for i in range(args.warmup + args.steps):
        b = i % w.batch
        kvh = (i // w.batch) % w.n_kv_heads
        dt, by, tk = oracle_sample(w, b, heads=range(kvh * G, kvh * G + G), threads=threads)
        if i >= args.warmup:
            times.append(dt)
            nbytes += by
            toks += tk
    total = sum(times)
    value = nbytes / total / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "kv_tokens_per_s": toks / total,
            "config": dict(w.describe(), sample="one request x one KV head group per step"),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": f"request i % {w.batch}, query heads of one KV head, "
                                       "append of that request + attention"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU arm
L2_BYTES = 129 * 10**6          # GB300 L2 (129 MB)
FLUSH_BYTES = 320 * 2**20       # > 2 x L2: written between timed launches when needed


def needs_flush(split_bytes: int) -> bool:
    """Working sets under ~2 x L2 are flushed between timed launches, so that
    every launch reads its cache from DRAM."""
    return split_bytes < 2 * L2_BYTES


class Case:
    """One workload made resident on the device: the cache prefilled through
    the library with every request's first L - q_len tokens, and the step's
    inputs (the last q_len tokens of each request, the queries)."""

    def __init__(self, F, w, ql, dev):
        import torch
        self.F, self.w, self.ql, self.dev = F, w, ql, dev
        nb, hkv, bs, d = w.num_blocks, w.n_kv_heads, w.block_size, w.head_dim
        ng = scale_groups(w)
        self.acc = accounting(w, q_len=ql)
        kc = torch.zeros((nb, hkv, bs, d), dtype=torch.uint8, device=dev)
        vc = None if w.mla else torch.zeros_like(kc)
        last_k, last_v = [], []
        self.seg_state = None
        if w.scale_mode == W.SCALE_CHANNEL_STATIC:
            kvs = [W.request_kv(w, b) for b in range(w.batch)]
            ks = F.kv_channel_scales(to_bf16_tensor(np.concatenate([k for k, _ in kvs]), dev),
                                     w.fmt)
            vs = F.kv_channel_scales(to_bf16_tensor(np.concatenate([v for _, v in kvs]), dev),
                                     w.fmt)
            get = lambda b: kvs[b]
        elif w.scale_mode == W.SCALE_SEGMENT:
            ks = torch.zeros((nb, F.segment_scale_heads(hkv)), dtype=torch.float32, device=dev)
            vs = None if w.mla else torch.zeros_like(ks)
            self.seg_state = torch.zeros((w.batch, 2, hkv, 2), dtype=torch.float32, device=dev)
            get = lambda b: W.request_kv(w, b)
        else:
            sdt = torch.uint8 if w.scale_mode == W.SCALE_MX_BLOCK else torch.float32
            ks = torch.zeros((nb, hkv, bs, ng), dtype=sdt, device=dev)
            vs = None if w.mla else torch.zeros_like(ks)
            get = lambda b: W.request_kv(w, b)
        self.prefill0 = None  # request 0's prefill rows (the bulk-append measurement)
        for b in range(w.batch):
            k, v = get(b)
            L = int(w.seq_lens[b])
            if L > ql:
                kd = to_bf16_tensor(k[:L - ql], dev)
                vd = None if v is None else to_bf16_tensor(v[:L - ql], dev)
                sd = torch.from_numpy(W.token_slots(w, b, 0, L - ql)).to(dev)
                if self.seg_state is not None:
                    F.kv_append_quant_segment(
                        kd, vd, sd, torch.tensor([0, L - ql], dtype=torch.int32, device=dev),
                        torch.zeros(1, dtype=torch.int32, device=dev), kc, vc, ks, vs,
                        self.seg_state[b:b + 1], fmt=w.fmt)
                else:
                    F.kv_append_quant(kd, vd, sd, kc, vc, ks, vs, fmt=w.fmt,
                                      scale_mode=w.scale_mode, group_size=w.group_size)
                if b == 0:
                    self.prefill0 = (kd, vd, sd)
            last_k.append(k[L - ql:L])
            if v is not None:
                last_v.append(v[L - ql:L])
        self.kc, self.vc, self.ks, self.vs = kc, vc, ks, vs
        self.vc_, self.vs_ = (kc, ks) if w.mla else (vc, vs)
        # step inputs, resident
        self.q_h = W.queries(w) if ql == 1 else W.chunk_queries(w, ql)
        self.kn_h = np.concatenate(last_k)
        self.vn_h = None if w.mla else np.concatenate(last_v)
        self.slot_h = np.concatenate([W.token_slots(w, b, int(w.seq_lens[b]) - ql,
                                                    int(w.seq_lens[b]))
                                      for b in range(w.batch)]).astype(np.int32)
        self.q = to_bf16_tensor(self.q_h, dev)
        self.kn = to_bf16_tensor(self.kn_h, dev)
        self.vn = None if w.mla else to_bf16_tensor(self.vn_h, dev)
        self.slots = torch.from_numpy(self.slot_h).to(dev)
        self.bt = torch.from_numpy(w.block_tables).to(dev)
        self.sl = torch.from_numpy(w.seq_lens).to(dev)
        oshape = (w.batch, w.n_q_heads, w.head_dim_v) if ql == 1 else \
            (w.batch, ql, w.n_q_heads, w.head_dim_v)
        self.out = torch.empty(oshape, dtype=torch.bfloat16, device=dev)
        self.ws = torch.empty(F.decode_workspace_bytes(w.batch, w.n_q_heads, hkv, d, w.head_dim_v,
                                                       bs, w.max_blocks, dev, q_len=ql),
                              dtype=torch.uint8, device=dev)
        if self.seg_state is not None:  # the step's varlen description
            self.seg_off = torch.arange(0, (w.batch + 1) * ql, ql, dtype=torch.int32, device=dev)
            self.seg_start = torch.from_numpy(w.seq_lens - ql).to(dev)

    def step(self, q=None, kn=None, vn=None, slots=None, sl=None):
        """One fp8pa_decode_step call: append (the split planner in the same
        launch), split kernel, merge.  The segment mode appends through its
        own call (it needs positions), then attends."""
        w = self.w
        if self.seg_state is not None:
            self.F.kv_append_quant_segment(self.kn if kn is None else kn,
                                           self.vn if vn is None else vn,
                                           self.slots if slots is None else slots, self.seg_off,
                                           self.seg_start, self.kc, self.vc, self.ks, self.vs,
                                           self.seg_state, fmt=w.fmt)
            attend = (self.F.paged_decode_attention if self.ql == 1
                      else self.F.paged_multiquery_attention)
            attend(self.q if q is None else q, self.kc, self.vc_, self.ks, self.vs_, self.bt,
                   self.sl if sl is None else sl, w.n_kv_heads, w.sm_scale, fmt=w.fmt,
                   scale_mode=w.scale_mode, group_size=w.group_size, head_dim_v=w.head_dim_v,
                   out=self.out, workspace=self.ws)
            return
        self.F.decode_step(self.kn if kn is None else kn, self.vn if vn is None else vn,
                           self.slots if slots is None else slots, self.q if q is None else q,
                           self.kc, self.vc_, self.ks, self.vs_, self.bt,
                           self.sl if sl is None else sl, w.n_kv_heads, w.sm_scale, fmt=w.fmt,
                           scale_mode=w.scale_mode, group_size=w.group_size,
                           head_dim_v=w.head_dim_v, out=self.out, workspace=self.ws)


def time_steps(case, steps, flush_buf, barrier):
    """Device time of `steps` decode steps (ms, the whole region), and of the
    split kernel inside each (ms per launch, CUDA events the library records
    on the call's stream around that launch).  With `flush_buf`, L2 is
    flushed before every step, outside the timed events."""
    import ctypes
    import torch
    from fp8_quantised_paged_gb300 import _native as N
    E = lambda: torch.cuda.Event(enable_timing=True)
    ev = [(E(), E()) for _ in range(steps)]
    for a, b_ in ev:  # materialise the event handles
        a.record()
        b_.record()
    torch.cuda.synchronize()
    if flush_buf is None:
        # Timed region 1: the steps back to back, nothing between launches.
        t0, t1 = E(), E()
        barrier()
        torch.cuda.synchronize()
        t0.record()
        for _ in range(steps):
            case.step()
        t1.record()
        torch.cuda.synchronize()
        barrier()
        ms_total = t0.elapsed_time(t1)
    else:
        st = [(E(), E()) for _ in range(steps)]
        barrier()
        torch.cuda.synchronize()
        for a, b_ in st:
            flush_buf.zero_()
            a.record()
            case.step()
            b_.record()
        torch.cuda.synchronize()
        barrier()
        ms_total = sum(a.elapsed_time(b_) for a, b_ in st)
    # Timed region 2: the same steps with the split launch bracketed.
    torch.cuda.synchronize()
    for i in range(steps):
        if flush_buf is not None:
            flush_buf.zero_()
        N.check(N.lib.fp8pa_set_split_events(ctypes.c_void_p(ev[i][0].cuda_event),
                                             ctypes.c_void_p(ev[i][1].cuda_event)), "events")
        case.step()
    torch.cuda.synchronize()
    N.check(N.lib.fp8pa_set_split_events(None, None), "events")
    return ms_total, [a.elapsed_time(b_) for a, b_ in ev]


def mla_on_tensor_cores(w) -> bool:
    """The latent layout runs the tcgen05 kernel for FP8 codes and query
    heads in groups of 64, the warp-MMA kernel otherwise."""
    return w.mla and w.fmt != W.INT8 and w.n_q_heads % 64 == 0


def chunk_on_tensor_cores(w, q_len: int) -> bool:
    """A causal chunk on the grouped-query layout runs the tcgen05 kernel for
    FP8 codes with one scale per (token, KV head), head_dim 128, block sizes
    16/32/64, when some qw dividing q_len gives 16 or 32 (query, head)
    columns per KV head."""
    g = w.n_q_heads // w.n_kv_heads
    return (not w.mla and w.fmt != W.INT8 and w.scale_mode == W.SCALE_TOKEN_HEAD
            and w.head_dim == 128 and w.head_dim_v == 128 and w.block_size in (16, 32, 64)
            and 2 <= q_len <= 8 and w.n_q_heads % w.n_kv_heads == 0
            and any(q_len % qw == 0 and g * qw in (16, 32) for qw in range(1, q_len + 1)))


def split_kernel_name(w, q_len: int = 1):
    if mla_on_tensor_cores(w):
        return "mla_tc_kernel", "decode_mla_tc.cu"
    if chunk_on_tensor_cores(w, q_len):
        return "gqa_tc_kernel", "decode_gqa_tc.cu"
    return ("mla_split_kernel", "decode_mla.cu") if w.mla else ("gqa_split_kernel", "decode_gqa.cu")


def split_roofline(w, acc, split_avg_ms, pk, traffic_json, q_len: int = 1):
    kname, src = split_kernel_name(w, q_len)
    # a causal chunk's capture is recorded under the workload's name + _q<len>
    traffic = traffic_per_launch(traffic_json, w.name if q_len == 1 else f"{w.name}_q{q_len}", src)
    if w.mla:
        # a dense contraction: tensor-bound; against the measured dense bf16
        # rate (the FP8 QK^T half could count against twice that: bf16 is
        # the conservative denominator)
        fl = flops_per_step(w)
        achieved = fl / (split_avg_ms * 1e-3) / 1e12
        return {"kernel": kname, "bound": "tensor", "achieved": achieved,
                "peak": pk["bf16_tflops"], "unit": "TFLOP/s", "frac": achieved / pk["bf16_tflops"],
                "traffic": traffic, "algorithmic_flops_per_launch": fl,
                "algorithmic_bytes_per_launch": acc["split"],
                "hbm_gbs_of_launch": acc["split"] / (split_avg_ms * 1e-3) / 1e9,
                "hbm_frac_of_launch": acc["split"] / (split_avg_ms * 1e-3) / 1e9 / pk["hbm_gbs"],
                "avg_launch_ms": split_avg_ms,
                "peak_source": pk["source"] + " (MEASURED_PEAKS.json bf16_tflops, burst)"}
    achieved = acc["split"] / (split_avg_ms * 1e-3) / 1e9
    return {"kernel": kname, "bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"],
            "unit": "GB/s", "frac": achieved / pk["hbm_gbs"], "traffic": traffic,
            "algorithmic_bytes_per_launch": acc["split"], "avg_launch_ms": split_avg_ms,
            "peak_source": pk["source"] + " (MEASURED_PEAKS.json hbm_gbs, copy bandwidth)"}


def append_roofline(case, launches, pk, traffic_json):
    """The bulk (prefill) append: request 0's first L - q_len tokens appended
    again (same slots, same values) `launches` times back to back from a CUDA
    graph, timed with CUDA events around the replay.  Algorithmic bytes = bf16 rows read + codes and scales
    written + slots read."""
    import torch
    w, F = case.w, case.F
    if case.prefill0 is None or case.seg_state is not None:
        return None
    kd, vd, sd = case.prefill0
    n = int(sd.numel())
    ntens = 1 if w.mla else 2
    per_row = w.head_dim * 2 + w.head_dim  # bf16 in, codes out
    if w.scale_mode == W.SCALE_TOKEN_HEAD:
        per_row += 4
    elif w.scale_mode == W.SCALE_TOKEN_GROUP:
        per_row += 4 * (w.head_dim // w.group_size)
    elif w.scale_mode == W.SCALE_MX_BLOCK:
        per_row += w.head_dim // w.group_size
    nbytes = n * ntens * w.n_kv_heads * per_row + 4 * n
    def call():
        F.kv_append_quant(kd, vd, sd, case.kc, case.vc, case.ks, case.vs, fmt=w.fmt,
                          scale_mode=w.scale_mode, group_size=w.group_size)
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    # The calls are captured once in a CUDA graph and replayed, so the launches
    # run back to back on the device and the events time the kernels, not the
    # host's per-call overhead (which is longer than one launch here).
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(launches):
            call()
    graph.replay()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    graph.replay()
    t1.record()
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / launches
    del graph
    achieved = nbytes / (ms * 1e-3) / 1e9
    try:
        with open(traffic_json) as f:
            t = json.load(f).get("append:" + w.name)
        traffic = (float(t["dram_bytes_per_launch"])
                   if t and t.get("kernel_source_sha256") == kernel_source_sha("append.cu")
                   else None)
    except (OSError, ValueError, KeyError, TypeError):
        traffic = None
    return {"kernel": "append_kernel", "bound": "hbm", "achieved": achieved,
            "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": achieved / pk["hbm_gbs"],
            "traffic": traffic, "algorithmic_bytes_per_launch": nbytes, "avg_launch_ms": ms,
            "tokens": n, "launches": launches,
            "what": f"bulk prefill append of request 0: {n} tokens x {w.n_kv_heads} KV heads x "
                    f"{ntens} tensor(s), bf16 in, {w.describe()['kv_fmt']} codes + scales out",
            "peak_source": pk["source"] + " (MEASURED_PEAKS.json hbm_gbs, copy bandwidth)"}


def run_gpu(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    import fp8_quantised_paged_gb300 as F

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = bench_workload(args)
    ql = args.q_len
    if ql > 1:
        args.no_cpu_baseline = True  # the oracle sample is a one-query decode
    pk = peaks()
    case = Case(F, w, ql, dev)
    acc = case.acc
    flush = needs_flush(acc["split"])
    flush_buf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev) if flush else None

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(args.warmup):
        case.step()
    torch.cuda.synchronize()
    assert F.get_device_error() == 0, "device error during warm-up"

    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    ms_total, split_ms = time_steps(case, args.steps, flush_buf, barrier)
    clk = clocks.stop()
    ms_total = max_over_ranks(ms_total, dev)
    ms_step = ms_total / args.steps
    assert F.get_device_error() == 0, "device error during the timed region"

    # ---- end to end through the public API with pinned host buffers
    e2e = e2e_plain = None
    if not args.no_e2e:
        # The step's inputs (q, new K/V rows, slots, lengths) are staged in
        # one pinned host buffer and copied in one transfer to a device
        # buffer holding the same layout, as a serving loop would.
        parts = [case.q_h.view(np.uint8).reshape(-1), case.kn_h.view(np.uint8).reshape(-1),
                 None if w.mla else case.vn_h.view(np.uint8).reshape(-1),
                 case.slot_h.view(np.uint8).reshape(-1), w.seq_lens.view(np.uint8).reshape(-1)]
        offs, total = [], 0
        for a in parts:
            offs.append(total)
            total += 0 if a is None else (a.size + 255) // 256 * 256
        host = torch.zeros(total, dtype=torch.uint8).pin_memory()
        hv = host.numpy()
        for o, a in zip(offs, parts):
            if a is not None:
                hv[o:o + a.size] = a
        dbuf = torch.empty(total, dtype=torch.uint8, device=dev)

        def dview(k, dtype, shape):
            n = int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
            return dbuf[offs[k]:offs[k] + n].view(dtype).view(shape)
        qd = dview(0, torch.bfloat16, case.q.shape)
        knd = dview(1, torch.bfloat16, case.kn.shape)
        vnd = None if w.mla else dview(2, torch.bfloat16, case.vn.shape)
        slotd = dview(3, torch.int32, case.slots.shape)
        sld = dview(4, torch.int32, case.sl.shape)
        out_p = torch.empty(case.out.shape, dtype=torch.bfloat16).pin_memory()
        h2d = total
        d2h = out_p.numel() * 2

        def e2e_body():
            dbuf.copy_(host, non_blocking=True)
            case.step(qd, knd, vnd, slotd, sld)
            out_p.copy_(case.out, non_blocking=True)

        def timed(fn):
            for _ in range(args.warmup):
                fn()
            barrier()
            t0 = time.perf_counter()
            for _ in range(args.steps):
                fn()
            return max_over_ranks((time.perf_counter() - t0) / args.steps, dev)

        # (1) plain calls: every step is the copy in, the fp8pa_decode_step
        # call (host-side validation, tensor maps, launches) and the copy out,
        # then a host synchronisation.
        def plain_step():
            e2e_body()
            torch.cuda.current_stream().synchronize()
        s_plain = timed(plain_step)
        # (2) a serving loop with fixed shapes captures the same sequence once
        # in a CUDA graph and replays it every step.
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            e2e_body()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            e2e_body()

        def graph_step():
            graph.replay()
            torch.cuda.current_stream().synchronize()
        s_graph = timed(graph_step)
        e2e = {"value": world * acc["step"] / s_graph / 1e9, "unit": "GB/s",
               "ms_per_step": s_graph * 1e3, "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h),
               "how": "CUDA graph of one pinned H2D copy, fp8pa_decode_step and one D2H copy "
                      "into pinned memory, replayed and host-synchronised every step"}
        e2e_plain = {"value": world * acc["step"] / s_plain / 1e9, "unit": "GB/s",
                     "ms_per_step": s_plain * 1e3, "h2d_bytes_per_step": int(h2d),
                     "d2h_bytes_per_step": int(d2h),
                     "how": "plain calls: pinned H2D copy, fp8pa_decode_step through the Python "
                            "binding (validation, tensor maps, launches), D2H copy, host "
                            "synchronisation, every step"}
        assert F.get_device_error() == 0, "device error in the e2e runs"

    app = None if args.no_append_roofline else append_roofline(case, min(args.steps, 50), pk,
                                                                args.traffic_json)
    split_avg_ms = statistics.mean(split_ms)
    roof = split_roofline(w, acc, split_avg_ms, pk, args.traffic_json, ql)
    del case
    flush_buf = None
    torch.cuda.empty_cache()

    # ---- the other workloads (each timed the same way, split kernel alone)
    per_workload = None
    if (not args.no_per_workload and ql == 1 and not args.mx_block and args.kv_fmt is None
            and args.scale_mode is None):
        per_workload = {}
        for idx in (3, 4, 5):
            if idx == args.workload:
                continue
            wi = W.make_workload(idx, "full")
            ci = Case(F, wi, 1, dev)
            fb = (torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
                  if needs_flush(ci.acc["split"]) else None)
            for _ in range(max(3, min(args.warmup, 5))):
                ci.step()
            torch.cuda.synchronize()
            n = max(5, min(args.steps, 20))
            tot, sp = time_steps(ci, n, fb, barrier)
            assert F.get_device_error() == 0, f"device error in workload {idx}"
            r = split_roofline(wi, ci.acc, statistics.mean(sp), pk, args.traffic_json)
            per_workload[wi.name] = {
                "config": dict(wi.describe(),
                               l2=("flushed (a 320 MiB write) before every step"
                                   if fb is not None else "no flush: cache larger than 2 x L2")),
                "steps": n, "ms_per_step": tot / n,
                "value": ci.acc["step"] / (tot / n * 1e-3) / 1e9, "unit": "GB/s",
                "kv_tokens_per_s": ci.acc["kv_tokens"] / (tot / n * 1e-3),
                "roofline": r}
            del ci, fb
            torch.cuda.empty_cache()

    if rank != 0:
        return
    value = world * acc["step"] / (ms_step * 1e-3) / 1e9
    kname = roof["kernel"]
    line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "pct_of_peak_hbm": 100.0 * value / world / pk["hbm_gbs"],
            "kv_tokens_per_s": world * acc["kv_tokens"] / (ms_step * 1e-3),
            "config": dict(w.describe(), parallelism=f"replicas x{world}",
                           kv_dtype={W.E4M3: "e4m3", W.E5M2: "e5m2", W.INT8: "int8"}[w.fmt],
                           compute=("fp8 codes: QK^T as tcgen05 FP8 MMAs (q as two E4M3 "
                                    "terms), P.V as tcgen05 bf16 MMAs (V^ and P as bf16 hi + lo), "
                                    "f32 accumulation in TMEM, f32 softmax"
                                    if mla_on_tensor_cores(w) else
                                    "fp8 codes: QK^T as tcgen05 FP8 MMAs (q as two E4M3 terms), "
                                    "P.V as tcgen05 f16 MMAs (V^ exact f16, P' as f16 hi + lo), "
                                    "f32 accumulation in TMEM, f32 softmax"
                                    if chunk_on_tensor_cores(w, ql) else
                                    ("int8" if w.fmt == W.INT8 else "fp8")
                                    + " codes -> exact f16, warp MMA (m16n8k16), f32 accumulate "
                                      "and softmax"),
                           l2=("flushed (a 320 MiB write) before every step, outside the timed "
                               "events" if flush else
                               "no flush: every step reads the whole cache, larger than 2 x L2"),
                           step=(f"fp8pa_kv_append_quant_segment ({ql} token(s)/request), "
                                 "then attention: plan, split, merge"
                                 if w.scale_mode == W.SCALE_SEGMENT else
                                 f"fp8pa_decode_step: append ({ql} token(s)/request) and plan, "
                                 "split, merge"),
                           q_len=ql,
                           bytes_per_step=acc["step"]),
            "roofline": roof,
            "append_roofline": app,
            "per_workload": per_workload,
            "gpu_launches": (4 if w.scale_mode == W.SCALE_SEGMENT else 3) * args.steps,
            "gpu_launches_per_step": (
                {"segment_append_kernel": 1, "plan_kernel": 1, kname: 1, "merge_kernel": 1}
                if w.scale_mode == W.SCALE_SEGMENT else
                {"append_plan_kernel": 1, kname: 1, "merge_kernel": 1}),
            "clocks": clk,
            "e2e": e2e,
            "e2e_plain_call": e2e_plain}
    if not args.no_cpu_baseline:
        import oracle
        threads = oracle.max_threads()
        G = w.n_q_heads // w.n_kv_heads
        dt, by, _ = oracle_sample(w, 0, heads=range(0, G), threads=threads)
        line["cpu_baseline"] = {"value": by / dt / 1e9, "unit": "GB/s", "cores": threads,
                                "kind": "oracle",
                                "sample": "request 0: append of its tokens + attention of the "
                                          f"{G} query heads of KV head 0 ({dt:.2f} s)"}
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        run_gpu(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
