#!/usr/bin/env python
"""Throughput of the quantized shared-KV sparse MLA attention forward on GB300.

One step = one pass of the whole hot path over one batch: qsfm_metadata
(split plan), the attention kernel and the combine kernel (launched only
when the plan may split tokens). Default workload: the CSA decode batch
(B = 128 sequences, S1 = 2 query tokens each, 64 heads x 512, S2 ~ U[4K, 64K],
cmp_ratio 4, K2 = 512 top-k indices, fp8 e4m3 KV with per-64 fp32 scales,
128-token pages). Metric: query tokens per second.

  python bench.py [--gpus N --steps K --warmup W] [--impl qsfm|reference]
                  [--workload I] [--kv-format fp8_fp32_scales|packed640|bf16]
                  [--n1 64|128] [--quick]

--kv-format and --n1 time the same workload with another KV row format or
head count (the default line is fp8 rows with fp32 scales and 64 heads).

Under torchrun each rank runs its own replica of the batch (no collective on
the data path); the step time is the max over ranks and the value counts the
tokens of all ranks (weak scaling). Rank 0 prints one JSON line.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

# the oracle's workers each use one BLAS thread (set before numpy loads)
os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
os.environ.setdefault("MKL_NUM_THREADS", "1")

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "query-tokens/s (64 heads, D=512) and % of roofline (HBM GB/s, TC util)"
UNIT = "query-tokens/s"
FLUSH_BYTES = 512 << 20  # > 129 MB L2
# bytes one KV row takes in each row format: 512 fp8 + 8 fp32 scales; a
# packed 640-byte row; 512 bf16
KV_ROW_BYTES = {"fp8_fp32_scales": 512 + 8 * 4, "packed640": 640, "bf16": 1024}
FLOPS_PER_ROW_HEAD = 4 * 512  # QK^T + PV per attended (token, row) and head
KERNEL_SRCS = [os.path.join(ROOT, "compressed_mla_attention_gb300", "csrc", f)
               for f in ("qsfm_attention.cu", "qsfm_device.cuh")]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "attention_traffic.txt")


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(values, device=None):
    """Element-wise max of `values` over all ranks (the step time of a weak
    scaling run is its slowest rank); identity without a process group."""
    dist = torch.distributed
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def job_throughput(world: int, tokens_per_rank: int, ms: float) -> float:
    """Query tokens per second of the whole job: every rank runs its own
    replica of the batch, so all ranks' tokens count, over the slowest
    rank's step time."""
    return world * tokens_per_rank / (ms / 1e3)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def kernel_sha() -> str:
    """Hash of the attention kernel's sources (its file and the device header
    it inlines): a recorded traffic figure holds only for this hash."""
    h = hashlib.sha256()
    for path in KERNEL_SRCS:
        h.update(open(path, "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: int):
    """DRAM bytes per attention launch from the committed ncu summary, or
    None when absent or taken on a different kernel source."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    sha = kernel_sha()
    for line in open(TRAFFIC_FILE):
        m = re.match(r"\s*workload=(\d+)\s+kernel_sha=(\w+)\s+dram_bytes_per_launch=(\d+)", line)
        if m and int(m.group(1)) == workload and m.group(2) == sha:
            return int(m.group(3))
    return None


# ------------------------------------------------------------ CPU baseline
def oracle_throughput(w, tokens, processes, min_seconds):
    """Query tokens/s of the fp64 oracle over `tokens`, repeated for at least
    min_seconds, on `processes` forked workers (call before CUDA init)."""
    from oracle import qsfm_oracle as O

    passes, t0 = 0, time.perf_counter()
    while True:
        O.reference_parallel(w, tokens, processes)
        passes += 1
        el = time.perf_counter() - t0
        if el >= min_seconds:
            return passes * len(tokens) / el, passes, el


# ------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------- GPU arm
def algorithmic_work(Q, p, w, dev):
    """Unique KV rows per batch and attended (token, row) pairs, counted from
    the rows the kernel resolves (exported debug gather)."""
    T = w.total_t
    max_rows = 2048
    tb = w.token_batch()
    per_batch = {}
    pairs = 0
    chunk = 64
    for lo in range(0, T, chunk):
        toks = torch.arange(lo, min(T, lo + chunk), dtype=torch.int32, device=dev)
        n = toks.numel()
        ids = torch.empty(n, max_rows, dtype=torch.int32, device=dev)
        counts = torch.empty(n, dtype=torch.int32, device=dev)
        Q.debug_gather(p, toks, max_rows, None, None, ids, counts)  # row ids only
        torch.cuda.synchronize()
        ids, counts = ids.cpu().numpy(), counts.cpu().numpy()
        for i in range(n):
            v = ids[i, :min(int(counts[i]), max_rows)]
            v = v[v >= 0]
            pairs += v.size
            per_batch.setdefault(int(tb[lo + i]), []).append(v)
    uniq = sum(np.unique(np.concatenate(v)).size for v in per_batch.values())
    return uniq, pairs


def run_gpu_arm(args, w, rank, world, local):
    import compressed_mla_attention_gb300 as Q

    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    a = W.device_inputs(w, dev)
    lse_wanted = a.pop("return_softmax_lse")
    out = torch.empty_like(a["q"])
    lse = torch.empty(w.total_t, w.n1, dtype=torch.float32, device=dev) if lse_wanted else None
    plan = torch.empty(1024, dtype=torch.int32, device=dev)
    p = Q.make_params(attn_out=out, softmax_lse=lse, metadata=plan, return_lse=lse_wanted,
                      num_ctas=args.ctas, **a)
    ws_bytes = Q.workspace_size(p)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    split = ws_bytes > 0
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        Q.metadata(p, plan, stream)
        if ev is not None:
            ev[1].record(stream)
        Q.attention(p, ws, stream)
        if ev is not None:
            ev[2].record(stream)
        if split:
            Q.combine(p, ws, stream)
        if ev is not None:
            ev[3].record(stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    if Q.device_status() != 0:
        raise RuntimeError("device fault during warm-up")

    # Timed steps: events only before and after each step, so that the
    # kernels of a step follow each other on the stream as in use (the
    # attention and combine kernels may start while their predecessor ends).
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    if not args.quick:
        clocks.start()
        time.sleep(0.3)
    for k in range(args.steps):
        flush.zero_()  # L2 flush, outside the timed events
        evs[k][0].record(stream)
        step()
        evs[k][1].record(stream)
    torch.cuda.synchronize()
    clk = None if args.quick else clocks.stop()
    if world > 1:
        torch.distributed.barrier()
    t_step = [e[0].elapsed_time(e[1]) for e in evs]
    # Per-kernel times (for the roofline of the attention kernel): a second
    # pass with events between the kernels.
    n_split = min(args.steps, 500)
    kevs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n_split)]
    for k in range(n_split):
        flush.zero_()
        step(kevs[k])
    torch.cuda.synchronize()
    t_plan = [e[0].elapsed_time(e[1]) for e in kevs]
    t_attn = [e[1].elapsed_time(e[2]) for e in kevs]
    t_comb = [e[2].elapsed_time(e[3]) for e in kevs]
    ms = statistics.mean(t_step)
    ms_attn = statistics.mean(t_attn)
    ms, ms_attn = max_over_ranks([ms, ms_attn], dev)
    if Q.device_status() != 0:
        raise RuntimeError("device fault during the timed steps")

    res = dict(ms=ms, ms_attn=ms_attn, ms_plan=statistics.mean(t_plan),
               ms_comb=statistics.mean(t_comb) if split else None,  # no combine launch
               launches=args.steps * (3 if split else 2), split=split, clocks=clk,
               ctas=int(plan[1].item()))

    # ---- end to end through the public API with pinned host buffers
    if not args.quick:
        host = {}
        for k_, v in a.items():
            if isinstance(v, torch.Tensor) and k_ not in ("ori_kv", "ori_scale", "cmp_kv", "cmp_scale"):
                host[k_] = v.cpu().pin_memory()
        out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = out_host.numel() * out_host.element_size() + (lse.numel() * 4 if lse_wanted else 0)
        lse_host = torch.empty(lse.shape, dtype=torch.float32).pin_memory() if lse_wanted else None
        dev_in = {k_: torch.empty_like(v, device=dev) for k_, v in host.items()}
        n_e2e = min(args.steps, 200)

        def e2e_step():
            # this step's inputs from pinned host memory, the public API call,
            # and the result read back to pinned host memory
            for k_, v in host.items():
                dev_in[k_].copy_(v, non_blocking=True)
            kw = dict(a)
            kw.update(dev_in)
            o, l = Q.quant_sparse_flash_mla(out=out, return_softmax_lse=lse_wanted, num_ctas=args.ctas, **kw)
            out_host.copy_(o, non_blocking=True)
            if lse_wanted:
                lse_host.copy_(l, non_blocking=True)

        def timed(run):
            times = []
            for k in range(args.warmup + n_e2e):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(torch.cuda.current_stream())
                run()
                e1.record(torch.cuda.current_stream())
                e1.synchronize()
                if k >= args.warmup:
                    times.append(e0.elapsed_time(e1))
            return statistics.mean(times)

        eager_ms = timed(e2e_step)
        # The same step captured once in a CUDA graph and replayed: the
        # copies and kernels of a step without the host's per-call launch
        # work (the library's calls are stream-ordered and capturable).
        graph_ms = None
        try:
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                for _ in range(3):
                    e2e_step()
            torch.cuda.current_stream().wait_stream(side)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                e2e_step()
            graph_ms = timed(graph.replay)
        except Exception as exc:  # capture unsupported here: the eager number stands
            print(f"e2e graph capture failed: {exc}", file=sys.stderr)
        e2e_ms = graph_ms if graph_ms is not None else eager_ms
        e2e_ms, eager_ms = max_over_ranks([e2e_ms, eager_ms], dev)
        res["e2e"] = dict(ms=e2e_ms, eager_ms=eager_ms, graph=graph_ms is not None, h2d=h2d, d2h=d2h)
    res["work"] = algorithmic_work(Q, p, w, dev)
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="qsfm", choices=["qsfm", "reference"])
    ap.add_argument("--workload", type=int, default=2)
    ap.add_argument("--kv-format", default="fp8_fp32_scales", choices=sorted(KV_ROW_BYTES),
                    help="KV row format of the workload (default: fp8 rows + fp32 scales)")
    ap.add_argument("--n1", type=int, default=64, choices=[64, 128], help="query heads")
    ap.add_argument("--ctas", type=int, default=0, help="planned CTAs (0 = SM count)")
    ap.add_argument("--quick", action="store_true", help="kernels only: no e2e, clocks, baseline")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--profile-size", action="store_true",
                    help="the CSA decode batch with S2 ~ U[4K, 8K] (for ncu captures)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local = dist_env()
    if args.impl == "reference" and rank != 0:
        return  # the CPU oracle arm runs on rank 0 only
    if world > 1 and args.impl == "qsfm":
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")

    w = W.profile_case() if args.profile_size else W.config(args.workload, kv_format=args.kv_format,
                                                             n1=args.n1)
    T = w.total_t
    cores = os.cpu_count() or 1

    if args.impl == "reference":
        from oracle import qsfm_oracle as O

        # calibrate one token, then size each step to keep the run short
        t0 = time.perf_counter()
        O.reference(w, [0])
        per_tok = time.perf_counter() - t0
        n = int(max(1, min(T, 90.0 * cores / max(per_tok, 1e-4) / (args.steps + args.warmup))))
        toks = W.subset_tokens(w, n, seed=7).tolist()
        for _ in range(args.warmup):
            O.reference_parallel(w, toks, min(cores, n))
        t0 = time.perf_counter()
        for _ in range(args.steps):
            O.reference_parallel(w, toks, min(cores, n))
        el = time.perf_counter() - t0
        v = args.steps * n / el
        line = {
            "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": w.name, "tokens_per_step": n, "parallelism": "none (CPU oracle)"},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": min(cores, n), "kind": "oracle",
                             "sample": f"{n} of the {T} query tokens per step, fp64 numpy oracle on "
                                       f"{min(cores, n)} forked workers"},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }
        print(json.dumps(line), flush=True)
        return

    # CPU baseline before CUDA initialises (the oracle pool forks)
    cpu = None
    if rank == 0 and world == 1 and not args.quick:
        tps, passes, el = oracle_throughput(w, list(range(T)), cores, args.cpu_seconds)
        cpu = {"value": tps, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"all {T} query tokens of the workload, {passes} passes ({el:.1f} s), "
                         f"fp64 numpy oracle on {cores} forked workers"}

    if rank == 0:
        from compressed_mla_attention_gb300 import build

        build.build()
    if world > 1:
        torch.distributed.barrier()
    res = run_gpu_arm(args, w, rank, world, local)
    if rank != 0:
        return
    hbm, tf, kind = measured_peaks()
    value = job_throughput(world, T, res["ms"])
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": res["ms"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "query_tokens": T, "global_batch": w.batch * world,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "flushed between steps (512 MiB write, outside the timed events)",
                   "ctas": res["ctas"], "split_kv": res["split"]},
        "gpu_launches": res["launches"],
        "kernel_ms": {"metadata": res["ms_plan"], "attention": res["ms_attn"], "combine": res["ms_comb"]},
    }
    if "work" in res:
        uniq, pairs = res["work"]
        n1 = w.n1
        q_bytes = T * n1 * 512 * 2
        o_bytes = T * n1 * 512 * 2
        idx_bytes = T * w.k2 * 4
        lse_bytes = T * n1 * 4 if w.return_lse else 0
        alg_bytes = uniq * KV_ROW_BYTES[args.kv_format] + q_bytes + o_bytes + idx_bytes + lse_bytes
        flops = pairs * FLOPS_PER_ROW_HEAD * n1
        achieved = alg_bytes / (res["ms_attn"] / 1e3) / 1e9
        # the recorded ncu traffic is for the default format and head count
        default_shape = args.kv_format == "fp8_fp32_scales" and n1 == 64 and not args.profile_size
        line["roofline"] = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                            "frac": achieved / hbm,
                            "traffic": recorded_traffic(args.workload) if default_shape else None,
                            "peak_kind": kind, "algorithmic_bytes": alg_bytes,
                            "tensor_tflops": flops / (res["ms_attn"] / 1e3) / 1e12,
                            "tensor_frac": flops / (res["ms_attn"] / 1e3) / 1e12 / tf}
    if "e2e" in res:  # not in --quick runs
        e = res["e2e"]
        line["e2e"] = {"value": job_throughput(world, T, e["ms"]), "unit": UNIT,
                       "h2d_bytes_per_step": e["h2d"], "d2h_bytes_per_step": e["d2h"],
                       "cuda_graph": e["graph"],
                       "eager_value": job_throughput(world, T, e["eager_ms"])}
    if res["clocks"] is not None:
        line["clocks"] = res["clocks"]
    if cpu is not None:
        line["cpu_baseline"] = cpu
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
