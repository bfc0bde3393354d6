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


PER_STEP_KEYS = ("q", "ori_block_table", "cmp_block_table", "cmp_sparse_indices", "seqused_ori_kv",
                 "seqused_cmp_kv", "cmp_residual_kv", "cmp_topk_length", "cu_seqlens_q", "seqused_q",
                 "sinks", "cu_seqlens_ori_kv", "cu_seqlens_cmp_kv", "ori_sparse_indices", "ori_topk_length")


def _step_input_sets(a, n_sets: int, seed: int):
    """n_sets host copies of one step's per-step inputs (everything but the
    resident KV tensors). Sets after the first get a fresh q and block
    tables permuted over the same pools (a bijection of the pool's blocks),
    so consecutive steps read mostly different KV rows (each set touches
    about as many bytes as one step reads; three sets exceed L2)."""
    g = torch.Generator().manual_seed(seed)
    base = {k: a[k].cpu() for k in PER_STEP_KEYS if isinstance(a.get(k), torch.Tensor)}
    sets = [base]
    for _ in range(n_sets - 1):
        s = dict(base)
        s["q"] = torch.randn(base["q"].shape, generator=g).to(base["q"].dtype)
        for tk, pool in (("ori_block_table", "ori_kv"), ("cmp_block_table", "cmp_kv")):
            if tk in base:
                perm = torch.randperm(int(a[pool].shape[0]), generator=g).to(torch.int32)
                t = base[tk]
                s[tk] = torch.where(t >= 0, perm[t.clamp(min=0).long()], t)
        sets.append(s)
    return sets


def _pack(tensors, align=256, pin=True):
    """One (pinned) byte buffer holding `tensors` back to back (256-byte
    aligned) and the (offset, nbytes, dtype, shape) of each."""
    layout, off = {}, 0
    for k, t in tensors.items():
        n = t.numel() * t.element_size()
        layout[k] = (off, n, t.dtype, tuple(t.shape))
        off += (n + align - 1) // align * align
    buf = torch.empty(max(off, align), dtype=torch.uint8)
    if pin:
        buf = buf.pin_memory()
    for k, t in tensors.items():
        o, n, _, _ = layout[k]
        buf[o:o + n].copy_(t.contiguous().view(-1).view(torch.uint8))
    return buf, layout


def _views(buf, layout):
    return {k: buf[o:o + n].view(dt).view(shape) for k, (o, n, dt, shape) in layout.items()}


def e2e_pipeline(Q, args, w, a, out, lse, lse_wanted, dev, world):
    """Query tokens/s through the public API (qsfm_metadata + qsfm_forward
    on parameter blocks made once per buffer slot) with every step's inputs
    uploaded from pinned host memory and its output read back to pinned
    host memory, pipelined over three streams: step k + 1's
    upload and step k - 1's read-back overlap step k's kernels (two device
    slots for inputs and outputs, events between the streams). Per step:
    one host-to-device copy of the packed inputs, one device-to-host copy
    of attn_out (and lse). The last two steps' outputs are checked bit for
    bit against quant_sparse_flash_mla run on the same inputs without the
    pipeline."""
    n_sets = 3
    sets = _step_input_sets(a, n_sets, seed=1234)
    packed = [_pack(s) for s in sets]
    layout = packed[0][1]
    h2d = packed[0][0].numel()
    slots_in = [torch.empty_like(packed[0][0], device=dev) for _ in range(2)]
    slots_out = [torch.empty_like(out) for _ in range(2)]
    slots_lse = [torch.empty_like(lse) for _ in range(2)] if lse_wanted else [None, None]
    host_out = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    host_lse = [torch.empty(lse.shape, dtype=torch.float32).pin_memory() for _ in range(2)] if lse_wanted \
        else [None, None]
    d2h = out.numel() * out.element_size() + (lse.numel() * 4 if lse_wanted else 0)
    s_c = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    fixed = {k: v for k, v in a.items() if k not in layout}
    # One parameter block, plan and workspace per slot, made once (a serving
    # loop's setup); every step is then the library's two calls,
    # qsfm_metadata() and qsfm_forward(), on the slot's buffers.
    plans = [torch.empty(Q.METADATA_INTS, dtype=torch.int32, device=dev) for _ in range(2)]
    params, wss = [], []
    for slot in range(2):
        kw = dict(fixed)
        kw.update(_views(slots_in[slot], layout))
        pp = Q.make_params(attn_out=slots_out[slot], softmax_lse=slots_lse[slot], metadata=plans[slot],
                           return_lse=lse_wanted, num_ctas=args.ctas, **kw)
        nb = Q.workspace_size(pp)
        params.append(pp)
        wss.append(torch.empty(nb, dtype=torch.uint8, device=dev) if nb else None)
    n = max(200, min(args.steps, 400))  # long enough that the pipeline's fill and drain are small

    def run(n_steps):
        ev_in = [torch.cuda.Event() for _ in range(n_steps)]
        ev_done = [torch.cuda.Event() for _ in range(n_steps)]
        ev_out = [torch.cuda.Event() for _ in range(n_steps)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(s_c)
        s_in.wait_stream(s_c)
        s_out.wait_stream(s_c)
        for k in range(n_steps):
            slot = k % 2
            if k >= 2:
                s_in.wait_event(ev_done[k - 2])  # step k - 2 has read this input slot
            with torch.cuda.stream(s_in):
                slots_in[slot].copy_(packed[k % n_sets][0], non_blocking=True)
                ev_in[k].record(s_in)
            s_c.wait_event(ev_in[k])
            if k >= 2:
                s_c.wait_event(ev_out[k - 2])  # step k - 2's output is read back
            Q.metadata(params[slot], plans[slot], s_c)
            Q.forward(params[slot], wss[slot], s_c)
            ev_done[k].record(s_c)
            s_out.wait_event(ev_done[k])
            with torch.cuda.stream(s_out):
                host_out[slot].copy_(slots_out[slot], non_blocking=True)
                if lse_wanted:
                    host_lse[slot].copy_(slots_lse[slot], non_blocking=True)
                ev_out[k].record(s_out)
        s_c.wait_event(ev_out[n_steps - 1])
        t1.record(s_c)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1)

    run(max(args.warmup, 3))
    ms = run(n) / n
    # result check: the last two steps again, kernels only, same inputs
    for k in (n - 2, n - 1):
        kw = dict(fixed)
        kw.update({kk: v.to(dev) for kk, v in sets[k % n_sets].items()})
        o, l = Q.quant_sparse_flash_mla(return_softmax_lse=lse_wanted, num_ctas=args.ctas, **kw)
        torch.cuda.synchronize()
        if not torch.equal(o.cpu(), host_out[k % 2]) or (lse_wanted and not torch.equal(l.cpu(), host_lse[k % 2])):
            raise RuntimeError(f"e2e step {k}: the read-back result differs from the kernels' result")
    (ms,) = max_over_ranks([ms], dev)
    return dict(ms=ms, h2d=h2d, d2h=d2h, n=n, sets=n_sets)


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
        res["e2e"] = e2e_pipeline(Q, args, w, a, out, lse, lse_wanted, dev, world)
    res["work"] = algorithmic_work(Q, p, w, dev)
    return res


def run_indexer(args, rank, world, local):
    """The lightning-indexer top-k (qsfm_lightning_indexer) on the call that
    feeds the CSA decode batch: K timed calls after W warm-up calls, L2
    flushed between calls, CUDA events on the launching stream. Algorithmic
    work: every batch's visible keys read once (128 e4m3 bytes + a 4-byte
    scale each) plus the queries, scales, weights and the index rows; FLOPs
    of the key-query products (2 per e4m3 pair) against the fp8 tensor peak
    (the measured bf16 peak times the nominal fp8 / bf16 ratio of 2)."""
    import compressed_mla_attention_gb300 as Q
    from compressed_mla_attention_gb300 import build

    build.build()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    w = W.indexer_decode_batch()
    a = W.indexer_device_inputs(w, dev)
    out = torch.empty(w.total_t, 1, w.topk, dtype=torch.int32, device=dev)
    ws = torch.empty(w.total_t * 32768 * 4, dtype=torch.uint8, device=dev)  # the largest score rows
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def call():
        Q.lightning_indexer(a["query"], a["query_scale"], a["weights"], a["key"], a["key_scale"],
                            a["block_table"], a["seqused_k"], layout=w.layout, batch=w.batch,
                            cmp_residual_k=a["cmp_residual_k"], topk=w.topk, mask_mode=w.mask_mode,
                            cmp_ratio=w.cmp_ratio, out=out, workspace=ws, stream=stream)

    for _ in range(args.warmup):
        flush.zero_()
        call()
    torch.cuda.synchronize()
    if Q.device_status() != 0:
        raise RuntimeError("device fault in the indexer warm-up")
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    for k in range(args.steps):
        flush.zero_()
        evs[k][0].record(stream)
        call()
        evs[k][1].record(stream)
    torch.cuda.synchronize()
    ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    # visible keys per token (the causal rule of the compressed keys)
    sk = w.seqused_k.numpy().astype(np.int64)
    res = w.cmp_residual_k.numpy().astype(np.int64) if w.cmp_residual_k is not None else np.zeros_like(sk)
    tb, tp = w.token_batch(), w.token_pos()
    s1 = w.q_lens[tb]
    pc = sk[tb] * w.cmp_ratio + res[tb] - s1 + tp
    vis = np.clip(np.floor_divide(pc + 1, w.cmp_ratio), 0, sk[tb]) if w.mask_mode == 3 else sk[tb]
    per_batch = np.zeros(w.batch, dtype=np.int64)
    np.maximum.at(per_batch, tb, vis)
    g = w.heads
    alg_bytes = int(per_batch.sum()) * (128 + 4) + w.total_t * (g * 128 + 2 * g * 4 + w.topk * 4)
    flops = int(vis.sum()) * g * 128 * 2
    hbm, tf, kind = measured_peaks()
    sec = ms / 1e3
    gbs, tfl = alg_bytes / sec / 1e9, flops / sec / 1e12
    hf, tcf = gbs / hbm, tfl / (2 * tf)
    line = {
        "metric": "indexer query-tokens/s (64 heads, d=128, top-512)", "value": w.total_t / sec,
        "unit": "query-tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 (fp32 accumulate)",
        "data": "synthetic",
        "config": {"workload": w.name, "query_tokens": w.total_t,
                   "l2": "flushed between calls (512 MiB write, outside the timed events)"},
        "gpu_launches": 2 * args.steps,  # score kernel + select kernel per call
        "roofline": {"bound": "tensor" if tcf > hf else "hbm", "frac": max(hf, tcf), "peak_kind": kind,
                     "hbm": {"achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": hf, "algorithmic_bytes": alg_bytes},
                     "tensor": {"achieved": tfl, "peak": 2 * tf, "unit": "TFLOP/s", "frac": tcf,
                                "algorithmic_flops": flops, "peak_note": "measured bf16 x 2 (nominal fp8 ratio)"},
                     "roofline_ms": max(alg_bytes / (hbm * 1e9), flops / (2 * tf * 1e12)) * 1e3},
    }
    print(json.dumps(line), flush=True)


def run_pipeline(args, rank, world, local):
    """The CSA decode step with its index rows made on the device (the CSA
    decode batch): per step the lightning indexer (score and select kernels)
    writes the index rows into the buffer the attention reads as
    cmp_sparse_indices, then the plan and the attention run on them. K timed
    steps after W warm-up steps, L2 flushed between steps outside the CUDA
    events on the launching stream; a second pass with events between the
    stages gives the indexer / plan + attention split."""
    import compressed_mla_attention_gb300 as Q
    from compressed_mla_attention_gb300 import build

    build.build()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    w = W.config(2)
    wi = W.indexer_for(w, seed=2)
    a = W.device_inputs(w, dev)
    a.pop("return_softmax_lse")
    ai = W.indexer_device_inputs(wi, dev)
    idx = torch.empty(w.total_t, 1, w.k2, dtype=torch.int32, device=dev)
    a["cmp_sparse_indices"] = idx
    ixws = torch.empty(w.total_t * 32768 * 4 + 4096, dtype=torch.uint8, device=dev)  # the largest score rows
    out = torch.empty_like(a["q"])
    plan = torch.empty(1024, dtype=torch.int32, device=dev)
    p = Q.make_params(attn_out=out, metadata=plan, num_ctas=args.ctas, **a)
    ws_bytes = Q.workspace_size(p)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    split = ws_bytes > 0
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step(ev=None):
        Q.lightning_indexer(ai["query"], ai["query_scale"], ai["weights"], ai["key"], ai["key_scale"],
                            ai["block_table"], ai["seqused_k"], layout=wi.layout, batch=wi.batch,
                            cmp_residual_k=ai["cmp_residual_k"], topk=wi.topk, mask_mode=wi.mask_mode,
                            cmp_ratio=wi.cmp_ratio, out=idx, workspace=ixws, stream=stream)
        if ev is not None:
            ev.record(stream)
        Q.metadata(p, plan, stream)
        Q.attention(p, ws, stream)
        if split:
            Q.combine(p, ws, stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    if Q.device_status() != 0:
        raise RuntimeError("device fault during the pipeline warm-up")
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    for k in range(args.steps):
        flush.zero_()
        evs[k][0].record(stream)
        step()
        evs[k][2].record(stream)
    torch.cuda.synchronize()
    ms = statistics.mean(e[0].elapsed_time(e[2]) for e in evs)
    for k in range(args.steps):
        flush.zero_()
        evs[k][0].record(stream)
        step(evs[k][1])
        evs[k][2].record(stream)
    torch.cuda.synchronize()
    if Q.device_status() != 0:
        raise RuntimeError("device fault during the timed pipeline steps")
    ms_ix = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    ms_att = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    line = {
        "metric": "CSA decode step with device-made index rows: query-tokens/s (indexer 64 heads top-512, "
                  "attention 64 heads D=512)",
        "value": w.total_t / (ms / 1e3), "unit": "query-tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3 indexer, f16 attention operands", "data": "synthetic",
        "config": {"workload": w.name, "indexer": wi.name, "query_tokens": w.total_t,
                   "l2": "flushed between steps (512 MiB write, outside the timed events)"},
        "stage_ms": {"indexer": ms_ix, "plan_attention_combine": ms_att},
        "gpu_launches": args.steps * (2 + (3 if split else 2)),
    }
    print(json.dumps(line), flush=True)


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
    ap.add_argument("--indexer", action="store_true",
                    help="time the lightning-indexer top-k on the call that feeds the CSA decode batch")
    ap.add_argument("--pipeline", action="store_true",
                    help="time the CSA decode step with its index rows made by the lightning indexer on the device")
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

    if args.indexer:
        if args.impl == "qsfm":
            run_indexer(args, rank, world, local)
        return
    if args.pipeline:
        if args.impl == "qsfm":
            run_pipeline(args, rank, world, local)
        return
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
        "vs_baseline": None, "dtype": "f16" if args.kv_format == "fp8_fp32_scales" else "bf16",
        "data": "synthetic",
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
        sec = res["ms_attn"] / 1e3
        gbs, tflops = alg_bytes / sec / 1e9, flops / sec / 1e12
        hbm_frac, tc_frac = gbs / hbm, tflops / tf
        # The roofline time is the slower of the two floors, max(bytes / HBM
        # peak, FLOPs / tensor peak); frac = that time / the measured time,
        # i.e. the larger of the two fractions, and `bound` names the floor
        # that sets it.
        tensor_bound = tc_frac > hbm_frac
        # the recorded ncu traffic is for the default format and head count
        default_shape = args.kv_format == "fp8_fp32_scales" and n1 == 64 and not args.profile_size
        line["roofline"] = {
            "bound": "tensor" if tensor_bound else "hbm",
            "achieved": tflops if tensor_bound else gbs,
            "peak": tf if tensor_bound else hbm,
            "unit": "TFLOP/s" if tensor_bound else "GB/s",
            "frac": max(hbm_frac, tc_frac),
            "traffic": recorded_traffic(args.workload) if default_shape else None,
            "peak_kind": kind,
            "hbm": {"achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": hbm_frac,
                    "algorithmic_bytes": alg_bytes},
            "tensor": {"achieved": tflops, "peak": tf, "unit": "TFLOP/s", "frac": tc_frac,
                       "algorithmic_flops": flops,
                       "dtype": "f16 operands (fp8 rows dequantised), fp32 accumulate"
                       if args.kv_format == "fp8_fp32_scales" else "bf16 operands, fp32 accumulate"},
            "roofline_ms": max(alg_bytes / (hbm * 1e9), flops / (tf * 1e12)) * 1e3,
            "kernel_ms": res["ms_attn"],
        }
    if "e2e" in res:  # not in --quick runs
        e = res["e2e"]
        line["e2e"] = {"value": job_throughput(world, T, e["ms"]), "unit": UNIT,
                       "h2d_bytes_per_step": e["h2d"], "d2h_bytes_per_step": e["d2h"],
                       "ms_per_step": e["ms"], "steps": e["n"],
                       "pipeline": "3 streams: upload k+1 | kernels k | read-back k-1; "
                                   f"{e['sets']} rotating input sets (fresh q, block tables permuted "
                                   "over the resident pools); last two results checked bitwise"}
    if res["clocks"] is not None:
        line["clocks"] = res["clocks"]
    if cpu is not None:
        line["cpu_baseline"] = cpu
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
