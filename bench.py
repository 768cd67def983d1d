"""Benchmark: paged decode / verify attention over a quantized paged KV cache.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

One step is one pass of the whole path over one synthetic batch: pa_plan
(device planner, plus the max|k_scale| reduction for per-channel scales),
pa_run (split-KV attention) and pa_combine (log-sum-exp merge), captured in a
CUDA graph and replayed.  The inputs are far larger than L2 (1.1-2.4 GB vs
129 MB); in addition, before every step a 256 MiB buffer is read (outside the
timed events) so that no line of the previous step survives in L2.  A read is
used rather than a write: written lines would be dirty, and writing them back
would land inside the next timed kernel.  `value` is the effective KV bandwidth: the bytes a
single pass must read (real tokens only, codes + scales, K and V once) divided
by the device time of the step.

By default every benchmark configuration is timed in turn and printed as one
JSON line each -- tiny fp16, bf16 GQA decode, E4M3 verify, INT8 and INT4
per-channel, and last, as the headline, the single-latent MQA batch (the
largest in tokens and in work).  --workload NAME times one of them (or the
verify / qsa workloads).  Before anything is timed, the oracle evaluates a
seeded sample of rows of the very batch about to be timed and the GPU output
must match it at the library's tolerances (the run fails otherwise); the
same oracle run's wall time is the line's cpu_baseline.  The latent workload
is a dense contraction: its roofline is the tensor rate (flops of S = q K^T
and O = P V over the visible tokens), with the HBM fraction beside it.

With N > 1 (torchrun, one rank per GPU) every rank times its own replica of
the batch (requests are independent, nothing is exchanged): weak scaling,
`value` is the sum over ranks of the bytes each processed / the slowest rank.

--op insert times the quantized paged KV insert instead (pa_insert): one
step writes 16384 new tokens (the largest step size of the Q pad + KV insert
measurements: B requests x next_n new tokens each) of the workload's shape
into its full-size pool, quantized to its encoding from rows in the query
dtype; `value` is the bytes the insert must move (new rows read, codes and
per-token scales written) divided by the step time.

--op sparse times sparse (selected-token) attention (pa_sparse_attention) on
the qsa workload: every query token attends to the positions its top-k
selection names; `value` is the K and V bytes of the selected tokens (each
query token and kv head reads its own) divided by the step time.

--impl reference times the CPU fp64 oracle on the host cores instead, each
step a bounded sample of rows of the same workload, in the same unit.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged-attn: effective KV HBM GB/s (% of GB300 peak) and query rows/sec"
WORKLOAD_TEXT = {
    "tiny": "tiny fp16 decode: B=2, L={37,70}, 4 q / 1 kv heads, D=64, bs=16, 12 blocks, fp32 out",
    "bf16": "bf16 GQA decode: B=64, L~U[512,8192], next_n=1, 32 q / 8 kv heads, D=128, bs=16, "
            "pool = pages + 10% slack, shuffled ids, bf16 out",
    "e4m3": "FP8 E4M3 verify: B=32, L~U[1024,32768], next_n=4 causal, 32 q / 8 kv heads, D=256, bs=32, "
            "per-tensor scales 0.05, NaN-poisoned null/slack/padding, bf16 out",
    "int8": "INT8 per-channel KV: B=128, L~U[2048,16384], next_n=1, 64 q / 8 kv heads, D=128, bs=16, "
            "k/v scales log-uniform [1e-2,1e3], q~N(0,100^2) fp16, fp32 out",
    "int4": "INT4 per-channel KV (packed 2/byte): B=128, L~U[2048,16384], next_n=1, 64 q / 8 kv heads, "
            "D=128, bs=16, k/v scales log-uniform [1e-2,1e3], q~N(0,100^2) fp16, fp32 out",
    "latent": "single-latent-KV MQA decode: B=256, L~lognormal(median 8192, sigma 1, cap 131072), next_n=2 "
              "causal, 128 q heads / 1 kv head, Dk=576, Dv=512 (first 512 of K), bs=64, E4M3 KV with a "
              "per-token fp32 scale, q~N(0,1) bf16, bf16 out",
    "verify": "FP8 E4M3 verify of 16 draft tokens: B=32, L~U[1024,32768], next_n=16 causal, 32 q / 8 kv heads "
              "(64 query rows per kv head), D=256, bs=32, per-tensor scales 0.05, NaN-poisoned null/slack/padding, "
              "bf16 out",
    "qsa": "sparse selected-token attention: 4 requests of 65536 tokens, 256 causal query rows each "
           "(1024 rows), 6 q / 1 kv heads, D=256, bs=16, fp16 KV, top-k 2048 selections, 90% shared "
           "per request, fp16 out",
}
SPARSE_TOP_K = 2048
FP4_TEXT = ("FP4 (MXFP4) paged MQA logits: B=128, L~U[4096,65536], next_n=2 causal, 64 heads, D=128 E2M1 with a "
            "UE8M0 scale per 32 values, bs=64 kv_fused blocks (68 B per token), per-head fp32 weights, bf16 logits "
            "[256, max_context_len]")
# the benchmark configurations in order; the last (largest in tokens and in
# work) is the headline line
ALL_CONFIGS = ("tiny", "bf16", "e4m3", "int8", "int4", "latent")
COMPUTE_DTYPE = {"tiny": "f16", "bf16": "bf16", "e4m3": "f16", "int8": "f16", "int4": "f16", "latent": "f16",
                 "qsa": "f16", "verify": "f16"}
L2_FLUSH_BYTES = 256 << 20


def _peaks(key: str = "hbm_gbs"):
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d[key]), "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}[key], "fallback"


# sources that decide each workload's attention kernel (traffic counters are
# only reported while these are unchanged)
KERNEL_SOURCES = {
    "latent": ("pa_latent.cu", "pa_attn.cuh", "pa_common.cuh", "pa_tc.cuh"),
    "fp4": ("pa_fp4.cu", "pa_attn.cuh", "pa_common.cuh"),
    "fp4_rectify": ("pa_fp4.cu", "pa_attn.cuh", "pa_common.cuh", "pa_tc.cuh"),
    "tiny": ("pa_attn.cuh", "pa_common.cuh", "pa_attn_launch.cuh", "pa_attn_f16_d64.cu"),
    "bf16": ("pa_attn.cuh", "pa_common.cuh", "pa_attn_launch.cuh", "pa_attn_bf16_d128.cu"),
    "e4m3": ("pa_e4m3_tc.cu", "pa_attn.cuh", "pa_common.cuh", "pa_tc.cuh"),
    "verify": ("pa_e4m3_tc.cu", "pa_attn.cuh", "pa_common.cuh", "pa_tc.cuh"),
    "sparse": ("pa_sparse.cu",),
    "int8": ("pa_attn.cuh", "pa_common.cuh", "pa_attn_launch.cuh", "pa_attn_int8_d128.cu"),
    "int4": ("pa_attn.cuh", "pa_common.cuh", "pa_attn_launch.cuh", "pa_attn_int4_d128_merged.cu"),
}
KERNEL_SOURCES.update({"insert_" + k: ("pa_insert.cu",) for k in ("tiny", "bf16", "e4m3", "int8", "int4", "latent")})


def attention_kernel_name(w) -> str:
    """The kernel pa_run launches for a workload (the dispatch rule of the C
    library: E4M3 at head dim 256 with per-tensor or no scales, 16..64 query
    rows per kv head in multiples of 16 and blocks of 16..128 tokens run on the
    tensor-core kernel; the single-latent shape on the latent kernel; the rest
    on the grouped warp-level kernel)."""
    if w.v_is_k_prefix:
        return "pa_latent_kernel"
    R = (w.Hq // w.Hkv) * w.n
    if (w.kv_dtype == "e4m3" and w.Dk == 256 and w.Dv == 256 and w.k_scale_mode in ("none", "tensor")
            and w.v_scale_mode in ("none", "tensor") and R % 16 == 0 and 16 <= R <= 64 and w.bs in (16, 32, 64, 128)):
        return "pa_e4m3_tc_kernel"
    return "pa_attn_kernel"


def _kernel_sha(workload: str) -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_attention_quantized_gb300", "csrc")
    for name in sorted(KERNEL_SOURCES[workload]):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def _traffic(workload: str):
    """DRAM bytes per attention launch from a committed ncu summary, only if it
    was taken on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)[workload]
        if d.get("kernel_sha") == _kernel_sha(workload):
            return d.get("dram_bytes_per_launch")
    except Exception:
        pass
    return None


def max_over_ranks(values, world: int, device):
    """Element-wise maximum of per-rank timings over all ranks (the slowest
    rank sets the step time); identity for one rank."""
    if world <= 1:
        return list(values)
    import torch
    import torch.distributed as dist
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_value(world: int, bytes_per_rank: int, ms_per_step: float) -> float:
    """Whole-job effective GB/s: every rank processes its own replica of the
    workload in the (max-over-ranks) step time."""
    return world * bytes_per_rank / (ms_per_step * 1e-3) / 1e9


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[2:6]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# new tokens per request of the insert step: 16384 new tokens in all
INSERT_NEW_TOKENS = {"tiny": 2, "bf16": 256, "e4m3": 512, "int8": 128, "int4": 128, "latent": 64}


def insert_bytes(w) -> int:
    """Algorithmic bytes of one insert: the new rows read (source dtype) plus
    the codes and per-token scales written."""
    rows = w.B * w.n * w.Hkv
    src = 2  # new rows in the query dtype (f16 / bf16)
    b = rows * (w.Dk * src + w.k_row_bytes + (4 if w.k_scale_mode == "token" else 0))
    if not w.v_is_k_prefix:
        b += rows * (w.Dv * src + w.v_row_bytes + (4 if w.v_scale_mode == "token" else 0))
    return b


# -------------------------------------------------------------- GPU arm


def gpu_arm(args, name, rank, world, local_rank, check=None):
    """Time workload `name`; `check(w, out, lse)` (rank 0) runs after one
    untimed pass and before anything is timed, and raises on a mismatch."""
    import torch
    import paged_attention_quantized_gb300 as pa
    from paged_attention_quantized_gb300 import build as pabuild
    from paged_attention_quantized_gb300 import workloads as W

    pabuild.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = W.make(name, device=dev, B=args.batch)
    p = pa.problem(w)
    out, lse, ws = pa.alloc(w, p, device=dev)
    B = pa.binding()
    eff_bytes = w.effective_kv_bytes()
    rows = w.B * w.n * w.Hq
    query_rows = w.B * w.n
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    s = torch.cuda.Stream(device=dev)
    launches_per_step = 3 if w.k_scale_mode == "channel" else 2
    launches_per_step += 1  # combine

    def dist_barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    # sanity before timing: no device error bits, every output finite
    with torch.cuda.stream(s):
        pa.run(w, p, out, ws, lse, stream=s)
    torch.cuda.synchronize()
    bits = B.pa_get_error(ws.data_ptr(), int(s.cuda_stream))
    if bits:
        raise RuntimeError(f"device error bits {bits:#x}")
    if not torch.isfinite(out.float()).all():
        raise RuntimeError("non-finite output")
    # correctness before timing: the oracle on sampled rows of this very batch
    extra = check(w, out, lse) if (check is not None and rank == 0) else {}
    dist_barrier()

    # capture one step
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pa.run(w, p, out, ws, lse, stream=s)
    torch.cuda.synchronize()

    def flush_l2():
        # evict the previous step's lines with clean ones (no write-back later)
        flush_sink.copy_(flush.view(torch.int64).sum())

    flush.fill_(1)
    flush_sink = torch.zeros((), dtype=torch.int64, device=dev)

    with torch.cuda.stream(s):
        for _ in range(args.warmup):
            flush_l2()
            g.replay()
    torch.cuda.synchronize()

    clocks = ClockSampler(int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local_rank)).split(",")[0])
                          if os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[0].isdigit() else local_rank)
    clocks.start()
    time.sleep(0.3)
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    dist_barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for k in range(args.steps):
            flush_l2()
            ev0[k].record(s)
            g.replay()
            ev1[k].record(s)
    torch.cuda.synchronize()
    dist_barrier()
    step_ms = [a.elapsed_time(b) for a, b in zip(ev0, ev1)]

    # the attention kernel alone, eager launches on the same stream
    a0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    a1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with torch.cuda.stream(s):
        for k in range(args.steps):
            flush_l2()
            pa.run(w, p, out, ws, lse, stream=s, steps="plan")
            a0[k].record(s)
            pa.run(w, p, out, ws, lse, stream=s, steps="run")
            a1[k].record(s)
            pa.run(w, p, out, ws, lse, stream=s, steps="combine")
    torch.cuda.synchronize()
    time.sleep(0.2)
    clk = clocks.stop()
    attn_ms = [a.elapsed_time(b) for a, b in zip(a0, a1)]

    # end to end through the public call with host buffers: q, block_table and
    # context_lens copied in from pinned memory, out copied back, every step
    hq = w.q.cpu().pin_memory()
    ht = w.block_table.cpu().pin_memory()
    hl = w.context_lens.cpu().pin_memory()
    ho = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        for _ in range(max(1, args.warmup)):
            w.q.copy_(hq, non_blocking=True)
            pa.run(w, p, out, ws, lse, stream=s)
    torch.cuda.synchronize()
    dist_barrier()
    e2e_ms = []
    with torch.cuda.stream(s):
        for k in range(args.steps):
            flush_l2()
            e0.record(s)
            w.q.copy_(hq, non_blocking=True)
            w.block_table.copy_(ht, non_blocking=True)
            w.context_lens.copy_(hl, non_blocking=True)
            pa.run(w, p, out, ws, lse, stream=s)
            ho.copy_(out, non_blocking=True)
            e1.record(s)
            e1.synchronize()
            e2e_ms.append(e0.elapsed_time(e1))
    h2d = hq.numel() * hq.element_size() + ht.numel() * 4 + hl.numel() * 4
    d2h = ho.numel() * ho.element_size()

    total_ms = sum(step_ms)
    attn_avg = sum(attn_ms) / len(attn_ms)
    e2e_avg = sum(e2e_ms) / len(e2e_ms)
    total_ms, attn_avg, e2e_avg = max_over_ranks([total_ms, attn_avg, e2e_avg], world, dev)
    ms_per_step = total_ms / args.steps
    value = job_value(world, eff_bytes, ms_per_step)
    peak, peak_kind = _peaks()
    achieved = eff_bytes / (attn_avg * 1e-3) / 1e9
    traffic = _traffic(name)
    roofline = {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": traffic,
                "kernel": attention_kernel_name(w), "peak_source": f"{peak_kind} hbm_gbs",
                "attn_ms": round(attn_avg, 5)}
    if w.v_is_k_prefix:
        # the latent path is a dense contraction: 2 (Dk + Dv) flops per
        # (query head row, visible token); f16 operands run at the bf16 rate
        L = w.context_lens.cpu().to(torch.int64)
        vis = sum(int((L - (w.n - 1 - j)).clamp(min=0).sum()) if w.causal else int(L.sum()) for j in range(w.n))
        flops = 2.0 * (w.Dk + w.Dv) * (w.Hq // w.Hkv) * vis
        tpeak, tkind = _peaks("bf16_tflops")
        tach = flops / (attn_avg * 1e-3) / 1e12
        roofline = {"bound": "tensor", "achieved": round(tach, 2), "peak": tpeak, "unit": "TFLOP/s",
                    "frac": round(tach / tpeak, 4), "traffic": traffic, "kernel": "pa_latent_kernel",
                    "peak_source": f"{tkind} bf16_tflops (f16 MMA, same rate)", "attn_ms": round(attn_avg, 5),
                    "flops_per_launch": flops,
                    "hbm": {"achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                            "frac": round(achieved / peak, 4)}}
    return {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "median_ms_per_step": round(statistics.median(step_ms), 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": COMPUTE_DTYPE[name],
        "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT[name] + ("" if args.batch is None else f" (batch {w.B})"),
                   "name": name, "batch": w.B,
                   "next_n": w.n, "total_tokens": int(w.context_lens.sum().item()),
                   "effective_kv_bytes": eff_bytes,
                   "l2": "inputs larger than L2; a 256 MiB buffer is read before every step to evict the "
                         "previous step's lines (clean, no write-back in the timed region)",
                   "parallelism": f"replicas x{world}"},
        "query_rows_per_s": round(world * query_rows / (ms_per_step * 1e-3), 1),
        "head_rows_per_s": round(world * rows / (ms_per_step * 1e-3), 1),
        "pct_of_hbm_peak": round(100.0 * value / world / peak, 2),
        "roofline": roofline,
        "e2e": {"value": round(world * eff_bytes / (e2e_avg * 1e-3) / 1e9, 2), "unit": "GB/s",
                "ms_per_step": round(e2e_avg, 5), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        **extra,
    }, w


def insert_arm(args, rank, world, local_rank):
    import torch
    import paged_attention_quantized_gb300 as pa
    from paged_attention_quantized_gb300 import build as pabuild
    from paged_attention_quantized_gb300 import workloads as W

    pabuild.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = W.make(args.workload, device=dev, B=args.batch, n=INSERT_NEW_TOKENS[args.workload])
    p = pa.problem(w)
    kn, vn = W.new_kv_rows(w, w.q_dtype, seed=w.seed + 100)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    nbytes = insert_bytes(w)
    tokens = w.B * w.n
    flush = torch.ones(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_sink = torch.zeros((), dtype=torch.int64, device=dev)
    s = torch.cuda.Stream(device=dev)

    def flush_l2():
        flush_sink.copy_(flush.view(torch.int64).sum())

    def dist_barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    with torch.cuda.stream(s):
        pa.insert(w, p, kn, vn, dev_error=err, stream=s)
    torch.cuda.synchronize()
    if int(err.item()):
        raise RuntimeError(f"device error bits {int(err.item()):#x}")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pa.insert(w, p, kn, vn, dev_error=err, stream=s)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for _ in range(args.warmup):
            flush_l2()
            g.replay()
    torch.cuda.synchronize()

    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    dist_barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for k in range(args.steps):
            flush_l2()
            ev0[k].record(s)
            g.replay()
            ev1[k].record(s)
    torch.cuda.synchronize()
    dist_barrier()
    step_ms = [a.elapsed_time(b) for a, b in zip(ev0, ev1)]
    # the kernel alone, eager launches on the same stream
    a0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    a1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with torch.cuda.stream(s):
        for k in range(args.steps):
            flush_l2()
            a0[k].record(s)
            pa.insert(w, p, kn, vn, dev_error=err, stream=s)
            a1[k].record(s)
    torch.cuda.synchronize()
    time.sleep(0.2)
    clk = clocks.stop()
    kern_ms = [a.elapsed_time(b) for a, b in zip(a0, a1)]

    # end to end: new rows, table and lengths in from pinned memory, the
    # error word back, every step
    hk = kn.cpu().pin_memory()
    hv = None if vn is None else vn.cpu().pin_memory()
    ht = w.block_table.cpu().pin_memory()
    hl = w.context_lens.cpu().pin_memory()
    he = torch.empty(1, dtype=torch.int32).pin_memory()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e2e_ms = []
    dist_barrier()
    with torch.cuda.stream(s):
        for k in range(args.steps):
            flush_l2()
            e0.record(s)
            kn.copy_(hk, non_blocking=True)
            if hv is not None:
                vn.copy_(hv, non_blocking=True)
            w.block_table.copy_(ht, non_blocking=True)
            w.context_lens.copy_(hl, non_blocking=True)
            pa.insert(w, p, kn, vn, dev_error=err, stream=s)
            he.copy_(err, non_blocking=True)
            e1.record(s)
            e1.synchronize()
            e2e_ms.append(e0.elapsed_time(e1))
    h2d = hk.numel() * hk.element_size() + (0 if hv is None else hv.numel() * hv.element_size()) + \
        ht.numel() * 4 + hl.numel() * 4
    total_ms, kern_avg, e2e_avg = max_over_ranks([sum(step_ms), sum(kern_ms) / len(kern_ms),
                                                  sum(e2e_ms) / len(e2e_ms)], world, dev)
    ms_per_step = total_ms / args.steps
    peak, peak_kind = _peaks()
    achieved = nbytes / (kern_avg * 1e-3) / 1e9
    line = {
        "metric": METRIC,
        "op": "insert",
        "value": round(job_value(world, nbytes, ms_per_step), 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "median_ms_per_step": round(statistics.median(step_ms), 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": f"quantized paged KV insert of {tokens} new tokens ({w.B} requests x {w.n}) into "
                               + WORKLOAD_TEXT[args.workload],
                   "name": args.workload, "batch": w.B, "new_tokens": tokens, "source_dtype": w.q_dtype,
                   "insert_bytes": nbytes,
                   "l2": "a 256 MiB buffer is read before every step to evict the previous step's lines",
                   "parallelism": f"replicas x{world}"},
        "tokens_per_s": round(world * tokens / (ms_per_step * 1e-3), 1),
        "pct_of_hbm_peak": round(100.0 * nbytes / (ms_per_step * 1e-3) / 1e9 / peak, 2),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": _traffic("insert_" + args.workload),
                     "kernel": "pa_insert_staged_kernel", "peak_source": f"{peak_kind} hbm_gbs",
                     "kernel_ms": round(kern_avg, 5)},
        "e2e": {"value": round(world * nbytes / (e2e_avg * 1e-3) / 1e9, 2), "unit": "GB/s",
                "ms_per_step": round(e2e_avg, 5), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": 4},
        "gpu_launches": args.steps,
        "clocks": clk,
    }
    return line, w, kn, vn


def selected_counts(w, sel) -> "list[int]":
    """Distinct visible positions each query token's selection names."""
    import numpy as np
    sl = sel.cpu().numpy()
    L = w.context_lens.cpu().numpy()
    out = []
    for b in range(w.B):
        for j in range(w.n):
            vis = int(L[b]) - (w.n - 1 - j) if w.causal else int(L[b])
            r = sl[b, j]
            out.append(int(np.unique(r[(r >= 0) & (r < vis)]).size))
    return out


def sparse_arm(args, rank, world, local_rank):
    import torch
    import paged_attention_quantized_gb300 as pa
    from paged_attention_quantized_gb300 import build as pabuild
    from paged_attention_quantized_gb300 import workloads as W

    pabuild.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = W.make(args.workload, device=dev, B=args.batch)
    sel = W.make_selection(w, k=SPARSE_TOP_K, seed=w.seed + 200, shared=0.9)
    p = pa.problem(w)
    B = pa.binding()
    ws = torch.zeros(max(256, B.pa_sparse_workspace_size(p, SPARSE_TOP_K)), dtype=torch.uint8, device=dev)
    out = torch.empty((w.B, w.n, w.Hq, w.Dv), dtype=pa.out_torch_dtype(w.out_dtype), device=dev)
    lse = torch.empty((w.B, w.n, w.Hq), dtype=torch.float32, device=dev)
    counts = selected_counts(w, sel)
    nbytes = sum(counts) * w.Hkv * (w.k_row_bytes + w.v_row_bytes)
    rows = w.B * w.n
    flush = torch.ones(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_sink = torch.zeros((), dtype=torch.int64, device=dev)
    s = torch.cuda.Stream(device=dev)

    def flush_l2():
        flush_sink.copy_(flush.view(torch.int64).sum())

    with torch.cuda.stream(s):
        pa.sparse_run(w, p, sel, out, ws, lse, stream=s)
    torch.cuda.synchronize()
    bits = B.pa_get_error(ws.data_ptr(), int(s.cuda_stream))
    if bits:
        raise RuntimeError(f"device error bits {bits:#x}")
    if not torch.isfinite(out.float()).all():
        raise RuntimeError("non-finite output")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pa.sparse_run(w, p, sel, out, ws, lse, stream=s)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for _ in range(args.warmup):
            flush_l2()
            g.replay()
    torch.cuda.synchronize()
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for k in range(args.steps):
            flush_l2()
            ev0[k].record(s)
            g.replay()
            ev1[k].record(s)
    torch.cuda.synchronize()
    step_ms = [a.elapsed_time(b) for a, b in zip(ev0, ev1)]
    # the call alone, eager, on the same stream (planner + attention)
    a0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    a1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with torch.cuda.stream(s):
        for k in range(args.steps):
            flush_l2()
            a0[k].record(s)
            pa.sparse_run(w, p, sel, out, ws, lse, stream=s)
            a1[k].record(s)
    torch.cuda.synchronize()
    time.sleep(0.2)
    clk = clocks.stop()
    call_ms = [a.elapsed_time(b) for a, b in zip(a0, a1)]
    # end to end: q, selections, table and lengths in from pinned memory, out back
    hq = w.q.cpu().pin_memory()
    hs = sel.cpu().pin_memory()
    ht = w.block_table.cpu().pin_memory()
    hl = w.context_lens.cpu().pin_memory()
    ho = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e2e_ms = []
    with torch.cuda.stream(s):
        for k in range(args.steps):
            flush_l2()
            e0.record(s)
            w.q.copy_(hq, non_blocking=True)
            sel.copy_(hs, non_blocking=True)
            w.block_table.copy_(ht, non_blocking=True)
            w.context_lens.copy_(hl, non_blocking=True)
            pa.sparse_run(w, p, sel, out, ws, lse, stream=s)
            ho.copy_(out, non_blocking=True)
            e1.record(s)
            e1.synchronize()
            e2e_ms.append(e0.elapsed_time(e1))
    h2d = hq.numel() * hq.element_size() + hs.numel() * 4 + ht.numel() * 4 + hl.numel() * 4
    d2h = ho.numel() * ho.element_size()
    total_ms, call_avg, e2e_avg = max_over_ranks([sum(step_ms), sum(call_ms) / len(call_ms),
                                                  sum(e2e_ms) / len(e2e_ms)], world, dev)
    ms_per_step = total_ms / args.steps
    peak, peak_kind = _peaks()
    achieved = nbytes / (call_avg * 1e-3) / 1e9
    return {
        "metric": METRIC,
        "op": "sparse",
        "value": round(job_value(world, nbytes, ms_per_step), 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "median_ms_per_step": round(statistics.median(step_ms), 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT[args.workload], "name": args.workload, "batch": w.B, "next_n": w.n,
                   "top_k": SPARSE_TOP_K, "selected_tokens": sum(counts), "selected_kv_bytes": nbytes,
                   "l2": "a 256 MiB buffer is read before every step to evict the previous step's lines",
                   "parallelism": f"replicas x{world}"},
        "query_rows_per_s": round(world * rows / (ms_per_step * 1e-3), 1),
        "pct_of_hbm_peak": round(100.0 * nbytes / (ms_per_step * 1e-3) / 1e9 / peak, 2),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": _traffic("sparse"), "kernel": "pa_sparse_attn_kernel",
                     "peak_source": f"{peak_kind} hbm_gbs", "call_ms": round(call_avg, 5),
                     "note": "timed over the whole call (planner + attention); selected rows shared between "
                             "the query tokens of a request can hit L2"},
        "e2e": {"value": round(world * nbytes / (e2e_avg * 1e-3) / 1e9, 2), "unit": "GB/s",
                "ms_per_step": round(e2e_avg, 5), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": 2 * args.steps,
        "clocks": clk,
    }, w, sel, nbytes


def fp4_arm(args, rank, world, local_rank):
    import torch
    import paged_attention_quantized_gb300 as pa
    from paged_attention_quantized_gb300 import build as pabuild
    from paged_attention_quantized_gb300 import workloads as W

    pabuild.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    kw = {} if args.batch is None else {"B": args.batch}
    w = W.make_fp4(device=dev, rectify=args.rectify, **kw)
    p = pa.fp4_problem(w)
    B = pa.binding()
    ws = torch.zeros(max(256, B.pa_fp4_logits_workspace_size(p)), dtype=torch.uint8, device=dev)
    out = torch.empty((w.B * w.n, w.max_context_len), dtype=torch.bfloat16, device=dev)
    nbytes = w.kv_bytes() + w.out_bytes()
    flush = torch.ones(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_sink = torch.zeros((), dtype=torch.int64, device=dev)
    s = torch.cuda.Stream(device=dev)

    def flush_l2():
        flush_sink.copy_(flush.view(torch.int64).sum())

    with torch.cuda.stream(s):
        pa.fp4_logits(w, p, out, ws, stream=s)
    torch.cuda.synchronize()
    bits = B.pa_get_error(ws.data_ptr(), int(s.cuda_stream))
    if bits:
        raise RuntimeError(f"device error bits {bits:#x}")
    extra = {}
    if rank == 0 and not args.no_cpu_baseline:
        extra = fp4_parity_and_baseline(w, out, args.cpu_baseline_s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pa.fp4_logits(w, p, out, ws, stream=s)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for _ in range(args.warmup):
            flush_l2()
            g.replay()
    torch.cuda.synchronize()
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for k in range(args.steps):
            flush_l2()
            ev0[k].record(s)
            g.replay()
            ev1[k].record(s)
    torch.cuda.synchronize()
    step_ms = [a.elapsed_time(b) for a, b in zip(ev0, ev1)]
    time.sleep(0.2)
    clk = clocks.stop()
    # end to end: q, scales, weights, table and lengths in from pinned memory, logits back
    hq, hs, hw = w.q.cpu().pin_memory(), w.sf_q.cpu().pin_memory(), w.weights.cpu().pin_memory()
    ht, hl = w.block_table.cpu().pin_memory(), w.context_lens.cpu().pin_memory()
    ho = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e2e_ms = []
    with torch.cuda.stream(s):
        for k in range(args.steps):
            flush_l2()
            e0.record(s)
            w.q.copy_(hq, non_blocking=True)
            w.sf_q.copy_(hs, non_blocking=True)
            w.weights.copy_(hw, non_blocking=True)
            w.block_table.copy_(ht, non_blocking=True)
            w.context_lens.copy_(hl, non_blocking=True)
            pa.fp4_logits(w, p, out, ws, stream=s)
            ho.copy_(out, non_blocking=True)
            e1.record(s)
            e1.synchronize()
            e2e_ms.append(e0.elapsed_time(e1))
    h2d = sum(t.numel() * t.element_size() for t in (hq, hs, hw, ht, hl))
    d2h = ho.numel() * ho.element_size()
    total_ms, e2e_avg = max_over_ranks([sum(step_ms), sum(e2e_ms) / len(e2e_ms)], world, dev)
    ms_per_step = total_ms / args.steps
    peak, peak_kind = _peaks()
    achieved = nbytes / (ms_per_step * 1e-3) / 1e9
    flops = 2.0 * 128 * w.H * sum(max(0, int(L) - (w.n - 1 - j)) for L in w.context_lens.tolist() for j in range(w.n))
    tpeak, tkind = _peaks("bf16_tflops")
    return {
        "metric": METRIC,
        "op": "fp4_logits",
        "value": round(job_value(world, nbytes, ms_per_step), 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "median_ms_per_step": round(statistics.median(step_ms), 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16",
        "data": "synthetic",
        "config": {"workload": FP4_TEXT + ("" if args.batch is None else f" (batch {w.B})")
                               + ("; each head's product clamped at 0 (per-head products on the tensor cores)"
                                  if args.rectify else "; plain weighted sum (heads folded into the query)"),
                   "name": "fp4" + ("_rectify" if args.rectify else ""), "rectify": bool(args.rectify),
                   "batch": w.B, "next_n": w.n, "total_tokens": int(w.context_lens.sum().item()),
                   "kv_bytes": w.kv_bytes(), "logit_bytes": w.out_bytes(),
                   "l2": "inputs larger than L2; a 256 MiB buffer is read before every step",
                   "parallelism": f"replicas x{world}"},
        "query_rows_per_s": round(world * w.B * w.n / (ms_per_step * 1e-3), 1),
        "pct_of_hbm_peak": round(100.0 * achieved / peak, 2),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": _traffic("fp4_rectify" if args.rectify else "fp4"),
                     "kernel": "pa_fp4_logits_kernel" if args.rectify else "pa_fp4_logits_sum_kernel",
                     "peak_source": f"{peak_kind} hbm_gbs",
                     "note": "timed over the whole call (plan, -inf fill, logits kernel); bytes = kv_fused of every "
                             "visible token once + the logits written",
                     "tensor": {"achieved": round(flops / (ms_per_step * 1e-3) / 1e12, 2), "peak": tpeak,
                                "unit": "TFLOP/s", "frac": round(flops / (ms_per_step * 1e-3) / 1e12 / tpeak, 4),
                                "peak_source": f"{tkind} bf16_tflops (f16 MMA, same rate)"}},
        "e2e": {"value": round(world * nbytes / (e2e_avg * 1e-3) / 1e9, 2), "unit": "GB/s",
                "ms_per_step": round(e2e_avg, 5), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": 3 * args.steps,
        "clocks": clk,
        **extra,
    }, w


def fp4_oracle_sample(w, budget_s: float, seed: int = 0):
    """The FP4 logits oracle on seeded query rows, about budget_s seconds."""
    import numpy as np
    from oracle import mqa_logits as OM
    wc = w.to("cpu")
    order = np.random.default_rng(seed).permutation(w.B * w.n)
    rows, outs = [], []
    t0 = time.perf_counter()
    for r in order:
        outs.append(OM.mqa_logits(wc, rows=[int(r)])[0])
        rows.append(int(r))
        if time.perf_counter() - t0 >= budget_s:
            break
    return rows, np.stack(outs), time.perf_counter() - t0


def fp4_parity_and_baseline(w, out, budget_s: float):
    """Oracle rows of the batch about to be timed: compared with the GPU's
    logits (same -inf / NaN pattern; |gpu - ref| <= 1e-2 * max(1, magnitude)
    for bf16 logits, the magnitude from the oracle on the sign-cleared inputs)
    before timing, and timed as the cpu_baseline."""
    import numpy as np
    from tests.test_fp4_gpu import magnitudes
    rows, ref, dt = fp4_oracle_sample(w, budget_s)
    mag = magnitudes(w, rows=rows)
    g = out[rows].float().cpu().numpy().astype(np.float64)
    if not (np.array_equal(np.isneginf(g), np.isneginf(ref)) and np.array_equal(np.isnan(g), np.isnan(ref))):
        raise RuntimeError("fp4 logits: masked / NaN columns differ from the oracle")
    fin = np.isfinite(ref)
    ratio = np.abs(g[fin] - ref[fin]) / np.maximum(1.0, mag[fin])
    if ratio.size and ratio.max() > 1e-2:
        raise RuntimeError(f"fp4 logits: error {ratio.max():.3g} of the magnitude exceeds 1e-2")
    L = w.context_lens.cpu().numpy()
    share = sum(int(L[r // w.n]) for r in rows) / float(w.n * L.sum())
    v = (w.kv_bytes() + w.out_bytes()) * share / dt / 1e9
    return {"parity": {"rows": len(rows), "of_rows": w.B * w.n, "max_err_over_magnitude": float(ratio.max(initial=0.0)),
                       "tol": 1e-2, "checked": "before timing, same batch"},
            "cpu_baseline": {"value": round(v, 5), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": f"{len(rows)} of {w.B * w.n} query rows, seeded, {dt:.1f} s, fp64 numpy; "
                                       f"GB/s scaled by the sampled share of the tokens; {cpu_model()}",
                             "query_rows_per_s": round(len(rows) / dt, 4)}}


def oracle_sparse_rate(w, sel, nbytes: int, budget_s: float, seed: int = 0):
    """Time the sparse oracle on a bounded sample of query tokens (all heads).
    Returns (GB/s equivalent, query rows/s, rows timed, seconds)."""
    import numpy as np
    from oracle import sparse as OS
    wc = w.to("cpu")
    sc = sel.cpu()
    rng = np.random.default_rng(seed)
    order = rng.permutation(w.B * w.n)
    n = 1
    while True:
        pick = order[:n]
        rows = [(int(r // w.n), int(r % w.n), h) for r in pick for h in range(w.Hq)]
        t0 = time.perf_counter()
        OS.sparse_attention(wc, sc, rows=rows)
        dt = time.perf_counter() - t0
        if dt >= budget_s / 4 or n >= w.B * w.n:
            break
        n = min(w.B * w.n, n * 2)
    share = n / (w.B * w.n)
    return nbytes * share / dt / 1e9, n / dt, n, dt


def oracle_insert_rate(w, kn, vn, budget_s: float):
    """Time the insert oracle on a bounded prefix of the requests.  Returns
    (GB/s equivalent, tokens/s, requests timed, seconds)."""
    from dataclasses import replace
    from oracle import insert as OI
    wc = w.to("cpu")
    # host pools written in place (the timed work is the insert, not a pool copy)
    wc = replace(wc, k_pool=wc.k_pool.numpy(), v_pool=None if wc.v_pool is None else wc.v_pool.numpy())
    kc = kn.cpu()
    vc = None if vn is None else vn.cpu()
    nb = 1
    while True:
        sub = replace(wc, B=nb, block_table=wc.block_table[:nb], context_lens=wc.context_lens[:nb])
        t0 = time.perf_counter()
        OI.insert(sub, kc[:nb], None if vc is None else vc[:nb], in_place=True)
        dt = time.perf_counter() - t0
        if dt >= budget_s / 4 or nb >= w.B:
            break
        nb = min(w.B, nb * 2)
    per_req = insert_bytes(w) / w.B
    return per_req * nb / dt / 1e9, nb * w.n / dt, nb, dt


# ---------------------------------------------------------- CPU oracle arm


def oracle_sample(w, budget_s: float, seed: int = 0, host=None):
    """Run the oracle on a bounded, seeded sample of (b, j, h) rows of
    workload w, sized to about budget_s seconds.  Returns (rows, out, lse,
    seconds of the timed run, threads, all rows)."""
    import numpy as np
    import oracle
    host = host if host is not None else oracle.HostArrays(w)
    threads = len(os.sched_getaffinity(0))
    allrows = np.stack(np.meshgrid(np.arange(w.B), np.arange(w.n), np.arange(w.Hq), indexing="ij"), -1).reshape(-1, 3)
    rng = np.random.default_rng(seed)
    perm = rng.permutation(len(allrows))
    # calibrate on a few rows, then size the sample to the budget
    n0 = min(len(allrows), max(threads, 8))
    t0 = time.perf_counter()
    oracle.attention(w, rows=allrows[perm[:n0]], host=host, threads=threads)
    dt = max(1e-6, time.perf_counter() - t0)
    n = int(min(len(allrows), max(n0, n0 * budget_s / dt)))
    rows = allrows[perm[:n]]
    t0 = time.perf_counter()
    ref, rlse = oracle.attention(w, rows=rows, host=host, threads=threads)
    dt = time.perf_counter() - t0
    return rows, ref, rlse, dt, threads, len(allrows)


def oracle_rate(w, budget_s: float, seed: int = 0):
    """Time the oracle on a bounded, seeded sample of rows of workload w.
    Returns (GB/s equivalent, rows/s, rows timed, seconds, threads)."""
    rows, _, _, dt, threads, nall = oracle_sample(w, budget_s, seed)
    n = len(rows)
    eff = w.effective_kv_bytes() * (n / nall)
    return eff / dt / 1e9, n / dt, n, dt, threads


def parity_and_baseline(w, out, lse, budget_s: float):
    """The oracle on a seeded sample of rows of the batch about to be timed:
    its wall time is the cpu_baseline, and its rows are compared with the
    GPU's output of the same batch at the library's tolerances (fp32 output
    2e-3, bf16 / fp16 1e-2; per-channel INT8 / INT4 normwise with the near-tie
    rule) -- a mismatch raises, so nothing is timed."""
    import oracle
    from tests.gpu_check import TOL, compare
    host = oracle.HostArrays(w)
    rows, ref, rlse, dt, threads, nall = oracle_sample(w, budget_s, host=host)
    n = len(rows)
    rep = {}
    compare(w, out, lse, rows=rows, host=host, report=rep, ref=(ref, rlse))
    v = w.effective_kv_bytes() * (n / nall) / dt / 1e9
    return {
        "parity": {"rows": n, "of_rows": nall, "max_abs_err": rep["max_err"], "tol": TOL[w.out_dtype],
                   "near_tie_hull_rows": rep["hull_rows"], "checked": "before timing, same batch",
                   "rule": "normwise |gpu-ref| <= tol * max(1, sum_t p_t |v_t|) with the near-tie hull"
                           if w.kv_dtype in ("int8", "int4") and w.k_scale_mode == "channel" else "max abs error"},
        "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"{n} of {nall} (b, j, h) rows, seeded, {dt:.1f} s; GB/s scaled by the "
                                   f"sampled share of the effective KV bytes; {cpu_model()}",
                         "query_rows_per_s": round(n / dt / w.Hq, 3)},
    }


REFERENCE_TOTAL_S = 150.0  # oracle seconds a whole reference run may take (all timed steps)


def ref_step_budget(args) -> float:
    """Oracle seconds per reference step: --ref-step-s, reduced so that the
    K timed steps together stay within REFERENCE_TOTAL_S."""
    return max(0.05, min(args.ref_step_s, REFERENCE_TOTAL_S / max(1, args.steps)))


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True).stdout
        for ln in out.splitlines():
            if ln.startswith("Model name"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


def reference_arm(args, name):
    from paged_attention_quantized_gb300 import workloads as W
    w = W.make(name, device="cpu", B=args.batch)
    for _ in range(args.warmup):
        oracle_rate(w, budget_s=0.5)
    vals, rows_s, secs = [], [], []
    n_rows = 0
    threads = 1
    for k in range(args.steps):
        v, r, n, dt, threads = oracle_rate(w, budget_s=ref_step_budget(args), seed=k)
        vals.append(v)
        rows_s.append(r)
        secs.append(dt)
        n_rows = n
    value = statistics.median(vals)
    total_rows = w.B * w.n * w.Hq
    sample = (f"{n_rows} of {total_rows} (b, j, h) rows per step, seeded; GB/s scaled by the sampled share "
              f"of the workload's effective KV bytes; {cpu_model()}")
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "GB/s",
        "n_gpus": args.gpus,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(1e3 * statistics.median(secs), 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT[name], "name": name},
        "query_rows_per_s": round(statistics.median(rows_s) / w.Hq, 3),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def reference_insert_arm(args):
    from paged_attention_quantized_gb300 import workloads as W
    w = W.make(args.workload, device="cpu", B=args.batch, n=INSERT_NEW_TOKENS[args.workload])
    kn, vn = W.new_kv_rows(w, w.q_dtype, seed=w.seed + 100)
    for _ in range(args.warmup):
        oracle_insert_rate(w, kn, vn, budget_s=0.2)
    vals, secs, toks = [], [], []
    nb = 1
    for _ in range(args.steps):
        v, r, nb, dt = oracle_insert_rate(w, kn, vn, budget_s=ref_step_budget(args))
        vals.append(v)
        secs.append(dt)
        toks.append(r)
    value = statistics.median(vals)
    return {
        "impl": "reference",
        "op": "insert",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "GB/s",
        "n_gpus": args.gpus,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(1e3 * statistics.median(secs), 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": f"quantized paged KV insert into {WORKLOAD_TEXT[args.workload]}",
                   "name": args.workload},
        "tokens_per_s": round(statistics.median(toks), 1),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"the first {nb} of {w.B} requests per step, single-threaded numpy; "
                                   f"{cpu_model()}"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def reference_fp4_arm(args):
    from paged_attention_quantized_gb300 import workloads as W
    kw = {} if args.batch is None else {"B": args.batch}
    w = W.make_fp4(device="cpu", rectify=args.rectify, **kw)
    L = w.context_lens.numpy()
    for _ in range(args.warmup):
        fp4_oracle_sample(w, budget_s=0.2)
    vals, secs, rs = [], [], []
    nr = 1
    for k in range(args.steps):
        rows, _, dt = fp4_oracle_sample(w, budget_s=ref_step_budget(args), seed=k)
        share = sum(int(L[r // w.n]) for r in rows) / float(w.n * L.sum())
        vals.append((w.kv_bytes() + w.out_bytes()) * share / dt / 1e9)
        secs.append(dt)
        rs.append(len(rows) / dt)
        nr = len(rows)
    value = statistics.median(vals)
    return {
        "impl": "reference",
        "op": "fp4_logits",
        "metric": METRIC,
        "value": round(value, 5),
        "unit": "GB/s",
        "n_gpus": args.gpus,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(1e3 * statistics.median(secs), 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": FP4_TEXT, "name": "fp4"},
        "query_rows_per_s": round(statistics.median(rs), 4),
        "cpu_baseline": {"value": round(value, 5), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{nr} of {w.B * w.n} query rows per step, seeded, fp64 numpy; {cpu_model()}"},
        "e2e": {"value": round(value, 5), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def reference_sparse_arm(args):
    from paged_attention_quantized_gb300 import workloads as W
    w = W.make(args.workload, device="cpu", B=args.batch)
    sel = W.make_selection(w, k=SPARSE_TOP_K, seed=w.seed + 200, shared=0.9)
    nbytes = sum(selected_counts(w, sel)) * w.Hkv * (w.k_row_bytes + w.v_row_bytes)
    for _ in range(args.warmup):
        oracle_sparse_rate(w, sel, nbytes, budget_s=0.2)
    vals, secs, rs = [], [], []
    nr = 1
    for k in range(args.steps):
        v, r, nr, dt = oracle_sparse_rate(w, sel, nbytes, budget_s=ref_step_budget(args), seed=k)
        vals.append(v)
        secs.append(dt)
        rs.append(r)
    value = statistics.median(vals)
    return {
        "impl": "reference",
        "op": "sparse",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "GB/s",
        "n_gpus": args.gpus,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(1e3 * statistics.median(secs), 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT[args.workload], "name": args.workload, "top_k": SPARSE_TOP_K},
        "query_rows_per_s": round(statistics.median(rs), 3),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{nr} of {w.B * w.n} query tokens (all heads) per step, seeded, fp64; "
                                   f"{cpu_model()}"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# -------------------------------------------------------------------- main


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="all", choices=["all"] + sorted(WORKLOAD_TEXT),
                    help="all (default): one line per benchmark configuration, the largest (latent) last")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ref-step-s", type=float, default=2.0, help="oracle seconds per reference step")
    ap.add_argument("--cpu-baseline-s", type=float, default=8.0,
                    help="oracle seconds (per configuration) for the parity check and cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--op", default="attention", choices=["attention", "insert", "sparse", "fp4"],
                    help="the step timed: the attention (default), the quantized paged KV insert, or sparse "
                         "selected-token attention (qsa workload)")
    ap.add_argument("--rectify", action="store_true",
                    help="--op fp4: clamp each head's product at 0 (per-head products, tensor cores)")
    ap.add_argument("--batch", type=int, default=None,
                    help="requests of the workload (default: its recipe); a smaller batch is for profiling only")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.op != "attention" and args.workload == "all":
        args.workload = {"sparse": "qsa", "insert": "bf16", "fp4": "bf16"}[args.op]   # the step's own workload
    names = ALL_CONFIGS if args.workload == "all" else (args.workload,)
    if args.impl == "reference":
        if rank != 0:
            return
        if args.op == "attention":
            saved = args.ref_step_s
            args.ref_step_s = saved / len(names)   # the whole run stays within a few minutes
            for name in names:
                print(json.dumps(reference_arm(args, name)), flush=True)
            args.ref_step_s = saved
            return
        arm = {"insert": reference_insert_arm, "sparse": reference_sparse_arm, "fp4": reference_fp4_arm}[args.op]
        print(json.dumps(arm(args)), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    if args.op == "fp4":
        line, w = fp4_arm(args, rank, world, local_rank)
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
            dist.destroy_process_group()
        if rank == 0:
            print(json.dumps(line), flush=True)
        return
    if args.op == "sparse":
        line, w, sel, nbytes = sparse_arm(args, rank, world, local_rank)
        if rank == 0 and not args.no_cpu_baseline:
            v, r, nr, dt = oracle_sparse_rate(w, sel, nbytes, args.cpu_baseline_s)
            line["cpu_baseline"] = {"value": round(v, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                                    "sample": f"{nr} of {w.B * w.n} query tokens (all heads), seeded, {dt:.1f} s, "
                                              f"fp64; GB/s scaled by the sampled share of the selected bytes; "
                                              f"{cpu_model()}",
                                    "query_rows_per_s": round(r, 3)}
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
            dist.destroy_process_group()
        if rank == 0:
            print(json.dumps(line), flush=True)
        return
    if args.op == "insert":
        line, w, kn, vn = insert_arm(args, rank, world, local_rank)
        if rank == 0 and not args.no_cpu_baseline:
            v, r, nb, dt = oracle_insert_rate(w, kn, vn, args.cpu_baseline_s)
            line["cpu_baseline"] = {"value": round(v, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                                    "sample": f"the first {nb} of {w.B} requests ({nb * w.n} new tokens), "
                                              f"{dt:.1f} s, single-threaded numpy; {cpu_model()}",
                                    "tokens_per_s": round(r, 1)}
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
            dist.destroy_process_group()
        if rank == 0:
            print(json.dumps(line), flush=True)
        return
    check = None if args.no_cpu_baseline else (lambda w, out, lse: parity_and_baseline(w, out, lse,
                                                                                      args.cpu_baseline_s))
    for name in names:
        line, w = gpu_arm(args, name, rank, world, local_rank, check=check)
        if len(names) > 1:
            line["headline"] = name == names[-1]
        del w
        if rank == 0:
            print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
