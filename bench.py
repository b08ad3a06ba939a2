"""Benchmark of the SDPA backward (and the NSA selected-attention backward).

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload 1..4]

Default workload 1: dense SDPA backward, fp16, b4 h12 s1024 d64, scale 1/8,
causal, BSHD storage viewed as BHSD (the GPT-2 sizes of the cuDNN-frontend
SDPA-backward sample).  A step is one sdpa_bwd call (preprocess, then the
main backward kernel, which also converts dQ) on inputs resident in HBM; the L2 is flushed between
steps by writing a 512 MB buffer outside the timed events.  FLOPs are
counted as 10 b h s_q s_kv d, halved for causal; NSA counts
10 T1 n1 (count * size) d over the selected slots.

Prints one JSON line (rank 0).  Under torchrun every rank runs its own
replica of the workload (independent problems, no data-path collective) and
value is the total over ranks divided by the slowest rank's time.
--impl reference times the fp64 CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import ctypes as C
import hashlib
import json
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "SDPA backward TFLOPS and fraction of GB300 FP16/BF16 tensor peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ------------------------------------------------------------------ workloads

def workload_info(idx):
    p = synth.workload(idx)
    if isinstance(p, synth.NsaProblem):
        flops = 10.0 * p.t1 * p.n1 * p.block_count * p.block_size * p.d
        name = (f"nsa_bwd_bf16_tnd_{len(p.cu_q)}x{p.t1 // len(p.cu_q)}_n1{p.n1}_n2{p.n2}_d{p.d}"
                f"_bs{p.block_size}x{p.block_count}_sparse{p.sparse_mode}")
        cfg = {"workload": name, "tokens": p.t1, "n1": p.n1, "n2": p.n2, "d": p.d, "block_size": p.block_size,
               "block_count": p.block_count, "sparse_mode": p.sparse_mode, "layout": "TND"}
        return p, flops, cfg
    lq = np.diff(np.concatenate([[0], p.cu_q]))
    lkv = np.diff(np.concatenate([[0], p.cu_kv]))
    flops = 10.0 * p.h * float((lq * lkv).sum()) * p.d * (0.5 if p.mask else 1.0)
    dt = "fp16" if p.dtype == synth.F16 else "bf16"
    if p.varlen:
        name = f"dense_bwd_{dt}_varlen{p.b}_h{p.h}_hkv{p.h_kv}_d{p.d}_causal_br_tnd"
        cfg = {"workload": name, "seqlens": [int(x) for x in lq], "h": p.h, "h_kv": p.h_kv, "d": p.d,
               "mask": "causal_bottom_right", "layout": "TND"}
    else:
        name = f"dense_bwd_{dt}_b{p.b}_h{p.h}_s{p.s_q}_d{p.d}_{'causal' if p.mask else 'full'}_bshd"
        cfg = {"workload": name, "b": p.b, "h": p.h, "h_kv": p.h_kv, "s_q": p.s_q, "s_kv": p.s_kv, "d": p.d,
               "scale": p.scale, "mask": ["none", "causal_top_left", "causal_bottom_right"][p.mask],
               "layout": "BSHD storage viewed as BHSD"}
    return p, flops, cfg


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "attention_backward_02_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def profile_traffic(kernel_tag):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel sources (profiles/<tag>.txt with source_hash and
    dram_bytes_per_launch lines); else None."""
    path = os.path.join(ROOT, "profiles", f"{kernel_tag}.txt")
    if not os.path.exists(path):
        return None
    vals = {}
    for line in open(path):
        if ":" in line:
            k, v = line.split(":", 1)
            vals[k.strip()] = v.strip()
    if vals.get("source_hash") != kernel_source_hash():
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ------------------------------------------------------------- clock sampling

class ClockSampler:
    """Polls NVML (the library nvidia-smi reads) for the SM clock and the
    clock-event reasons of one GPU while running; read-only."""

    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown",
               0x4: "sw_power_cap"}

    def __init__(self, pci_bus_id, period_s=0.002):
        self.samples, self.period, self.ok = [], period_s, False
        self._stop = threading.Event()
        try:
            self.nvml = C.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                return
            self.handle = C.c_void_p()
            if self.nvml.nvmlDeviceGetHandleByPciBusId_v2(pci_bus_id.encode(), C.byref(self.handle)) != 0:
                return
            self.reasons_fn = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(self.nvml, "nvmlDeviceGetCurrentClocksThrottleReasons")
            self.max_mhz = C.c_uint()
            self.nvml.nvmlDeviceGetMaxClockInfo(self.handle, 1, C.byref(self.max_mhz))  # NVML_CLOCK_SM
            self.ok = True
        except (OSError, AttributeError):
            return

    def _run(self):
        clk, reasons = C.c_uint(), C.c_ulonglong()
        while not self._stop.is_set():
            self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, C.byref(clk))
            self.reasons_fn(self.handle, C.byref(reasons))
            self.samples.append((clk.value, reasons.value))
            time.sleep(self.period)

    def __enter__(self):
        if self.ok:
            self.thread = threading.Thread(target=self._run, daemon=True)
            self.thread.start()
        return self

    def __exit__(self, *exc):
        if self.ok:
            self._stop.set()
            self.thread.join()

    def summary(self):
        if not self.ok or not self.samples:
            return None
        reasons = set()
        for _, r in self.samples:
            for bit, name in self.REASONS.items():
                if r & bit:
                    reasons.add(name)
        return {"sm_mhz": float(statistics.median(c for c, _ in self.samples)),
                "sm_max_mhz": float(self.max_mhz.value), "reasons": sorted(reasons),
                "samples": len(self.samples), "source": "NVML (nvidia-smi's library), polled every 2 ms"}


# ---------------------------------------------------------------- CPU oracle

def _last_rows(cu, n):
    """Indices of the last min(n, length) tokens of every sequence (inclusive cumulative lengths), and
    how many each sequence gave."""
    starts = np.concatenate([[0], cu[:-1]])
    take = np.minimum(cu - starts, n)
    idx = np.concatenate([np.arange(e - t, e) for e, t in zip(cu, take)]) if len(cu) else np.zeros(0, np.int64)
    return idx.astype(np.int64), take.astype(np.int64)


def oracle_dense_sample(p, rows=None):
    """The last `rows` query rows of every sequence, every head, against all of that sequence's keys.
    With bottom-right alignment each of those rows sees exactly the keys it sees in p (whose causal
    workloads have equal query and key lengths, or are bottom-right already).  Returns the callable,
    its FLOPs (10 d per visible pair, the metric's convention), a description and its (sequence,
    kv head) unit count."""
    import oracle
    idx, take = _last_rows(p.cu_q, p.s_q if rows is None else max(1, int(rows)))
    lkv = p.cu_kv - np.concatenate([[0], p.cu_kv[:-1]])
    q, do = p.f64("q")[idx], p.f64("do")[idx]
    k, v = p.f64("k"), p.f64("v")
    cu_q = np.cumsum(take)
    mask = oracle.CAUSAL_BOTTOM_RIGHT if p.mask else oracle.MASK_NONE
    o, lse = oracle.dense_fwd(q, k, v, cu_q, p.cu_kv, p.scale, mask)
    if p.mask:  # row i of a sequence's sample sees keys 0 .. i + (lkv - rows)
        pairs = sum(int(np.clip(np.arange(t) + (n - t) + 1, 0, n).sum()) for t, n in zip(take, lkv))
    else:
        pairs = int((take * lkv).sum())
    flops = 10.0 * p.h * pairs * p.d

    def run():
        oracle.dense_bwd(q, k, v, o, do, lse, cu_q, p.cu_kv, p.scale, mask)

    desc = f"last {int(take.max())} query rows of each of the {len(take)} sequences, all {p.h} heads, fp64"
    return run, flops, desc, len(take) * p.h_kv


def oracle_nsa_sample(p, tokens=None):
    """The last `tokens` query tokens of every sequence, all heads, against all of that sequence's keys
    (the selections and the sparse mode's bottom-right alignment as in p)."""
    import oracle
    idx, take = _last_rows(p.cu_q, p.t1 if tokens is None else max(1, int(tokens)))
    q, do, topk = p.f64("q")[idx], p.f64("do")[idx], p.topk[idx]
    k, v = p.f64("k"), p.f64("v")
    cu_q = np.cumsum(take)
    o, mx, sm = oracle.nsa_fwd(q, k, v, topk, cu_q, p.cu_kv, p.scale, p.block_size, p.sparse_mode)
    flops = 10.0 * float(take.sum()) * p.n1 * p.block_count * p.block_size * p.d

    def run():
        oracle.nsa_bwd(q, k, v, o, do, mx, sm, topk, cu_q, p.cu_kv, p.scale, p.block_size, p.sparse_mode)

    desc = f"last {int(take.max())} tokens of each of the {len(take)} sequences, all {p.n1} heads, fp64"
    return run, flops, desc, len(take) * p.n2


def cpu_sample(p, target_s):
    """A sample of the workload whose oracle run takes about target_s (at most the whole workload).
    Returns (run, flops, description, threads the oracle runs it on: one per (sequence, kv head) unit
    at most)."""
    import oracle
    build = oracle_nsa_sample if isinstance(p, synth.NsaProblem) else oracle_dense_sample
    full = p.t1 if isinstance(p, synth.NsaProblem) else p.s_q
    run, _, _, _ = build(p, 64)
    t0 = time.perf_counter(); run(); dt = time.perf_counter() - t0
    run, flops, desc, units = build(p, min(full, 64 * max(1.0, target_s / max(dt, 1e-6))))
    return run, flops, desc, max(1, min(oracle.thread_count(), units))


def affinity_count():
    """Host cores this process may run on (the oracle's threads use the online count)."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def time_repeated(run, min_s, max_runs=10000):
    """Calls run() until at least min_s seconds have passed (at least once); returns (runs, seconds)."""
    n, t0 = 0, time.perf_counter()
    while True:
        run()
        n += 1
        dt = time.perf_counter() - t0
        if dt >= min_s or n >= max_runs:
            return n, dt


def run_reference(args, info):
    import oracle
    p, _, cfg = info
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    per_step = min(30.0, 120.0 / max(1, args.steps + args.warmup))
    run, flops, desc, threads = cpu_sample(p, per_step)
    for _ in range(args.warmup):
        run()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter(); run(); times.append(time.perf_counter() - t0)
    total = sum(times)
    value = flops * args.steps / total / 1e12
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": cfg,
            "impl": "reference",
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "sample": desc, "affinity": affinity_count(), "host_threads": oracle.thread_count()},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------ rank arithmetic

def slowest_rank_ms(total_ms, dist=None, device="cpu"):
    """Max over ranks of a rank's summed step time: the replicas' job ends
    with its slowest rank.  dist: torch.distributed (initialised) or None."""
    if dist is None:
        return float(total_ms)
    import torch
    t = torch.tensor([float(total_ms)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world, flops_per_replica, ms_per_step):
    """Whole-job throughput: every replica's FLOPs over the slowest rank's time per step."""
    return world * flops_per_replica / (ms_per_step * 1e-3) / 1e12


# ------------------------------------------------------------------- GPU arm

def run_ours(args, info):
    import torch
    import attention_backward_02_gb300 as ab
    from tests import harness as H

    p, flops, cfg = info
    rank, world = int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    lib = ab._lib.load()
    stream = torch.cuda.current_stream()
    nsa = isinstance(p, synth.NsaProblem)

    # ---- inputs resident in HBM (O and the stats from the forward) ----
    if nsa:
        o_bits, mx, sm = H.nsa_oracle_inputs(p)
        q, k, v, do, o = (H.bits_to_gpu(x, p.dtype) for x in (p.q, p.k, p.v, p.do, o_bits))
        mx8 = torch.from_numpy(np.repeat(mx[..., None], 8, -1)).cuda()
        sm8 = torch.from_numpy(np.repeat(sm[..., None], 8, -1)).cuda()
        topk = torch.from_numpy(p.topk).cuda()
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        desc = H.nsa_desc(p)
        ws = torch.empty(ab.nsa_workspace_size(desc), dtype=torch.uint8, device="cuda")
        inputs = [q, k, v, o, do, mx8, sm8, topk]
        outputs = [dq, dk, dv]
        launches_per_step = 7

        def step():
            ab.nsa_selected_attn_bwd(desc, q, k, v, o, do, mx8, sm8, topk, dq, dk, dv, workspace=ws, stream=stream)
    else:
        q, k, v, do = (H.bits_to_gpu(x, p.dtype) for x in (p.q, p.k, p.v, p.do))
        o = torch.empty_like(q)
        lse = torch.empty(p.t_q * p.h, dtype=torch.float32, device="cuda")
        desc = H.dense_desc(p)
        vq, vk, vv, vo = H.dense_views(p, (q, k, v, o))
        ab.sdpa_fwd_stats(desc, vq, vk, vv, vo, lse)  # O and LSE from the library's forward
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        vdo, vdq, vdk, vdv = H.dense_views(p, (do, dq, dk, dv))
        ws = torch.empty(ab.sdpa_workspace_size(desc)[1], dtype=torch.uint8, device="cuda")
        inputs = [q, k, v, o, do, lse]
        outputs = [dq, dk, dv]
        launches_per_step = 2  # preprocess, main kernel (which also converts dQ)

        def step():
            ab.sdpa_bwd(desc, vq, vk, vv, vo, vdo, lse, vdq, vdk, vdv, workspace=ws, stream=stream)

    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    for _ in range(args.warmup):
        step()
        flush.fill_(1)
    assert ab.attn_query_status(ws) == 0, "device status flagged during warm-up"

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    for e in ev:  # instantiate the events before the timed region
        for x in e:
            x.record(stream)
    torch.cuda.synchronize()
    props = torch.cuda.get_device_properties(local)
    bus = getattr(props, "pci_bus_id", None)
    pci = (f"{getattr(props, 'pci_domain_id', 0):08x}:{getattr(props, 'pci_bus_id', 0):02x}:"
           f"{getattr(props, 'pci_device_id', 0):02x}.0") if bus is not None else "00000000:00:00.0"
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(pci) as clocks:
        t_wall = time.perf_counter()
        for i in range(args.steps):
            e_call0, _, _, e_call1 = ev[i]
            e_call0.record(stream)
            step()
            e_call1.record(stream)
            flush.fill_(1)  # L2 flush outside the timed events
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
    if dist:
        dist.barrier()
    # second pass, same steps: events around the main kernel alone (for the
    # roofline); events inside the call break the launch overlap, so this pass
    # does not feed the headline number
    for i in range(args.steps):
        _, e_main0, e_main1, _ = ev[i]
        lib.attn_set_main_kernel_events(C.c_void_p(e_main0.cuda_event), C.c_void_p(e_main1.cuda_event))
        step()
        lib.attn_set_main_kernel_events(None, None)
        flush.fill_(1)
    torch.cuda.synchronize()
    call_ms = [ev[i][0].elapsed_time(ev[i][3]) for i in range(args.steps)]
    main_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(args.steps)]
    total_ms = slowest_rank_ms(sum(call_ms), dist, "cuda")
    assert ab.attn_query_status(ws) == 0, "device status flagged during the timed steps"
    ms_per_step = total_ms / args.steps
    value = job_tflops(world, flops, ms_per_step)
    main_mean = statistics.mean(main_ms)

    # ---- warm L2: the same call back to back, no flush in between (context beside the flushed figure) ----
    warm_steps = max(1, min(args.steps, 50))
    w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    step()
    w0.record(stream)
    for _ in range(warm_steps):
        step()
    w1.record(stream)
    torch.cuda.synchronize()
    warm_ms = w0.elapsed_time(w1) / warm_steps

    # ---- end to end through the C ABI with host buffers ----
    host_in = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True).copy_(x) for x in inputs]
    host_out = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in outputs]
    h2d = sum(x.numel() * x.element_size() for x in host_in)
    d2h = sum(x.numel() * x.element_size() for x in host_out)
    e2e_steps = max(1, min(args.steps, 50))
    e2e_ms = []
    for i in range(e2e_steps):
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for dst, src in zip(inputs, host_in):
            dst.copy_(src, non_blocking=True)
        step()
        for dst, src in zip(host_out, outputs):
            dst.copy_(src, non_blocking=True)
        a1.record(stream)
        a1.synchronize()
        e2e_ms.append(a0.elapsed_time(a1))
        flush.fill_(1)
    e2e_val = job_tflops(world, flops, statistics.mean(e2e_ms))

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return
    pk, pk_src = peaks()
    peak = float(pk["bf16_tflops"])  # fp16 and bf16 share one dense rate
    achieved = flops / (main_mean * 1e-3) / 1e12
    tag = "nsa_bwd_main" if nsa else "dense_bwd_main"
    traffic = profile_traffic(f"{tag}_workload{args.workload}")
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "ms_per_step_median": statistics.median(call_ms),
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16" if p.dtype == synth.F16 else "bf16", "data": "synthetic",
        "config": dict(cfg, l2="flushed: 512 MB buffer written between timed steps, outside the events",
                       inputs="N(0,1) seeded; O and stats from the library forward" if not nsa else
                       "N(0,1) seeded; O and softmax stats from the oracle sparse forward",
                       parallelism=f"replicas x{world}" if world > 1 else "single GPU"),
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": tag, "kernel_ms": main_mean,
                     "peak_source": f"{pk_src} bf16_tflops (burst; fp16 has the same dense rate)",
                     "whole_call_frac": value / world / peak},
        "e2e": {"value": e2e_val, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": statistics.mean(e2e_ms)},
        "warm_l2": {"value": job_tflops(world, flops, warm_ms), "unit": "TFLOP/s", "ms_per_step": warm_ms,
                    "steps": warm_steps},
        "gpu_launches": launches_per_step * args.steps,  # of the timed pass
        "clocks": clocks.summary(),
        "wall_s_timed_region": t_wall,
    }
    if world == 1 and not args.no_cpu_baseline:
        import oracle
        run, cflops, desc_s, threads = cpu_sample(p, 10.0)
        nrun, dt = time_repeated(run, 10.0)  # about 10 s of CPU work, repeating a sample smaller than that
        line["cpu_baseline"] = {"value": cflops * nrun / dt / 1e12, "unit": "TFLOP/s", "cores": threads,
                                "host_threads": oracle.thread_count(),
                                "kind": "oracle", "sample": f"{desc_s}; run {nrun} time(s)", "seconds": dt,
                                "affinity": affinity_count()}
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=1, choices=[1, 2, 3, 4])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    info = workload_info(args.workload)
    if args.impl == "reference":
        run_reference(args, info)
    else:
        run_ours(args, info)


if __name__ == "__main__":
    main()
