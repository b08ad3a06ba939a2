"""Benchmark of the SDPA backward (and the NSA selected-attention backward).

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload 1..4]

Default workload 1: dense SDPA backward, fp16, b4 h12 s1024 d64, scale 1/8,
causal, BSHD storage viewed as BHSD (the GPT-2 sizes of the cuDNN-frontend
SDPA-backward sample).  A step is one sdpa_bwd call (preprocess, then the
main backward kernel, dQ finalize) on inputs resident in HBM; the L2 is flushed between
steps by writing a 512 MB buffer outside the timed events.  The line also carries the other
workloads (2-4, both dQ modes) under "workloads".  FLOPs are
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

def workload_info(idx, p=None):
    """(problem, FLOPs per step, config) of workload idx; p: a shard of it (default: the workload)."""
    p = synth.workload(idx) if p is None else p
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

def shard_seed(idx, rank):
    """Seed of rank `rank`'s shard of workload idx: rank 0 draws exactly the single-GPU workload."""
    return 42 + idx + 7919 * rank


def shard_units(per_rank_seqs, kv_heads, rank):
    """The (global sequence, kv head) units of rank `rank`'s shard.  The global problem holds
    world * per_rank_seqs sequences; rank r owns sequences [r * per_rank_seqs, (r + 1) *
    per_rank_seqs) with every kv head.  The units are independent (each owns its dQ / dK / dV rows),
    so the shards need no collective on the data path."""
    s0 = rank * per_rank_seqs
    return [(s, g) for s in range(s0, s0 + per_rank_seqs) for g in range(kv_heads)]


def shard_workload(idx, rank):
    """Rank `rank`'s shard of the global problem of workload idx: the workload's sequences, drawn
    with the rank's own seed (the sequences are the global ones [rank * b, (rank + 1) * b))."""
    return synth.workload(idx, seed=shard_seed(idx, rank)) if rank else synth.workload(idx)


def slowest_rank_ms(total_ms, dist=None, device="cpu"):
    """Max over ranks of a rank's summed step time: the sharded job ends
    with its slowest rank.  dist: torch.distributed (initialised) or None."""
    if dist is None:
        return float(total_ms)
    import torch
    t = torch.tensor([float(total_ms)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world, flops_per_replica, ms_per_step):
    """Whole-job throughput: every rank's shard's FLOPs (equal per rank) over the slowest rank's time
    per step."""
    return world * flops_per_replica / (ms_per_step * 1e-3) / 1e12


# ------------------------------------------------------------------- GPU arm

def nsa_useful_flops(p):
    """FLOPs of the selected slots whose block has at least one key the token sees under the sparse
    mode (10 d per visible-block key, n1 heads): the slot count less the fully masked filler blocks."""
    starts_q = np.concatenate([[0], p.cu_q[:-1]])
    lq = p.cu_q - starts_q
    lkv = p.cu_kv - np.concatenate([[0], p.cu_kv[:-1]])
    seq = np.repeat(np.arange(len(lq)), lq)
    pos = np.arange(p.t1) - starts_q[seq]
    if p.sparse_mode == 2:
        last = pos + (lkv - lq)[seq]                       # last visible key of each token
        first_key = p.topk.astype(np.int64) * p.block_size  # [T1, n2, cnt]
        useful = (first_key <= last[:, None, None]).sum()
    else:
        useful = p.topk.size
    return 10.0 * float(useful) * (p.n1 // p.n2) * p.block_size * p.d


class Problem:
    """One workload's inputs resident in HBM, its outputs and workspace, and step(set, stream): one
    backward call on buffer set `set` (two sets, for the pipelined end-to-end measurement)."""

    def __init__(self, p, deterministic, sets=1):
        import torch
        import attention_backward_02_gb300 as ab
        from tests import harness as H
        self.p, self.ab = p, ab
        self.nsa = isinstance(p, synth.NsaProblem)
        self.sets = []
        if self.nsa:
            self.desc = H.nsa_desc(p, deterministic)
            self.launches = 7
            nbytes = ab.nsa_workspace_size(self.desc)
            for si in range(sets):
                q, k, v, do = (H.bits_to_gpu(x, p.dtype) for x in (p.q, p.k, p.v, p.do))
                topk = torch.from_numpy(p.topk).cuda()
                if si == 0:  # O and the softmax stats from the library's sparse forward
                    o = torch.empty(p.t1, p.n1, p.v.shape[-1], dtype=q.dtype, device="cuda")
                    mx8 = torch.empty(p.t1, p.n1, 8, dtype=torch.float32, device="cuda")
                    sm8 = torch.empty_like(mx8)
                    fws = ab.nsa_selected_attn_fwd(H.nsa_desc(p), q, k, v, topk, o, mx8, sm8)
                    assert ab.attn_query_status(fws) == 0
                else:
                    o, mx8, sm8 = (self.sets[0]["inputs"][i].clone() for i in (3, 5, 6))
                dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
                ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
                self.sets.append(dict(inputs=[q, k, v, o, do, mx8, sm8, topk], outputs=[dq, dk, dv], ws=ws))
        else:
            self.desc = H.dense_desc(p, deterministic)
            self.launches = 3  # preprocess, main kernel, dQ finalize
            nbytes = ab.sdpa_workspace_size(self.desc)[1]
            for si in range(sets):
                q, k, v, do = (H.bits_to_gpu(x, p.dtype) for x in (p.q, p.k, p.v, p.do))
                if si == 0:
                    o = torch.empty_like(q)
                    lse = torch.empty(p.t_q * p.h, dtype=torch.float32, device="cuda")
                    vq, vk, vv, vo = H.dense_views(p, (q, k, v, o))
                    ab.sdpa_fwd_stats(H.dense_desc(p), vq, vk, vv, vo, lse)  # O and LSE from the library forward
                else:
                    o, lse = self.sets[0]["inputs"][3].clone(), self.sets[0]["inputs"][5].clone()
                dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
                ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
                views = H.dense_views(p, (q, k, v, o, do, dq, dk, dv))
                self.sets.append(dict(inputs=[q, k, v, o, do, lse], outputs=[dq, dk, dv], ws=ws, views=views))

    def step(self, si=0, stream=None):
        t = self.sets[si]
        if self.nsa:
            q, k, v, o, do, mx8, sm8, topk = t["inputs"]
            dq, dk, dv = t["outputs"]
            self.ab.nsa_selected_attn_bwd(self.desc, q, k, v, o, do, mx8, sm8, topk, dq, dk, dv, workspace=t["ws"],
                                          stream=stream)
        else:
            vq, vk, vv, vo, vdo, vdq, vdk, vdv = t["views"]
            self.ab.sdpa_bwd(self.desc, vq, vk, vv, vo, vdo, t["inputs"][5], vdq, vdk, vdv, workspace=t["ws"],
                             stream=stream)

    def status(self, si=0):
        return self.ab.attn_query_status(self.sets[si]["ws"])


def time_calls(prob, steps, flush, stream, lib):
    """Per step: CUDA events around the whole call (L2 flushed between steps, outside the events), then
    a second pass with events around the main kernel alone.  Returns (call_ms list, main_ms list)."""
    import torch
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    for e in ev:  # instantiate the events before the timed region
        for x in e:
            x.record(stream)
    torch.cuda.synchronize()
    for i in range(steps):
        e_call0, _, _, e_call1 = ev[i]
        e_call0.record(stream)
        prob.step(0, stream)
        e_call1.record(stream)
        flush.fill_(1)
    torch.cuda.synchronize()
    # events inside the call break the launch overlap, so this pass does not feed the headline number
    for i in range(steps):
        _, e_main0, e_main1, _ = ev[i]
        lib.attn_set_main_kernel_events(C.c_void_p(e_main0.cuda_event), C.c_void_p(e_main1.cuda_event))
        prob.step(0, stream)
        lib.attn_set_main_kernel_events(None, None)
        flush.fill_(1)
    torch.cuda.synchronize()
    return [ev[i][0].elapsed_time(ev[i][3]) for i in range(steps)], [ev[i][1].elapsed_time(ev[i][2]) for i in range(steps)]


def e2e_pipelined(prob, steps, flush_unused=None):
    """End to end through the C ABI with host buffers, steps pipelined over two device buffer sets and
    three streams: the host-to-device copy of step i+1 and the device-to-host copy of step i-1 overlap
    the call of step i.  Returns ms per step (first copy in to last copy out, over steps)."""
    import torch
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    host_in = [[torch.empty(x.shape, dtype=x.dtype, pin_memory=True).copy_(x) for x in t["inputs"]]
               for t in prob.sets]
    host_out = [[torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in t["outputs"]] for t in prob.sets]
    ev_in = [torch.cuda.Event() for _ in prob.sets]
    ev_cmp = [torch.cuda.Event() for _ in prob.sets]
    ev_out = [torch.cuda.Event() for _ in prob.sets]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(s_in)
    for i in range(steps):
        si = i % len(prob.sets)
        t = prob.sets[si]
        if i >= len(prob.sets):  # the set's previous step has been computed and copied out
            s_in.wait_event(ev_cmp[si])
            s_in.wait_event(ev_out[si])
        with torch.cuda.stream(s_in):
            for dst, src in zip(t["inputs"], host_in[si]):
                dst.copy_(src, non_blocking=True)
        ev_in[si].record(s_in)
        s_cmp.wait_event(ev_in[si])
        prob.step(si, s_cmp)
        ev_cmp[si].record(s_cmp)
        s_out.wait_event(ev_cmp[si])
        with torch.cuda.stream(s_out):
            for dst, src in zip(host_out[si], t["outputs"]):
                dst.copy_(src, non_blocking=True)
        ev_out[si].record(s_out)
    t1.record(s_out)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) / steps


def run_ours(args, info):
    import torch
    import attention_backward_02_gb300 as ab

    rank, world = int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    # this rank's shard of the global problem (rank 0: the workload itself); equal FLOPs on every rank
    p, flops, cfg = info if rank == 0 else workload_info(args.workload, shard_workload(args.workload, rank))
    if rank != 0:
        cfg = info[2]
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    lib = ab._lib.load()
    stream = torch.cuda.current_stream()
    nsa = isinstance(p, synth.NsaProblem)
    prob = Problem(p, False, sets=2)
    launches_per_step = prob.launches
    inputs, outputs = prob.sets[0]["inputs"], prob.sets[0]["outputs"]

    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    for _ in range(args.warmup):
        prob.step(0, stream)
        flush.fill_(1)
    assert prob.status() == 0, "device status flagged during warm-up"
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
        call_ms, main_ms = time_calls(prob, args.steps, flush, stream, lib)
        t_wall = time.perf_counter() - t_wall
    if dist:
        dist.barrier()
    total_ms = slowest_rank_ms(sum(call_ms), dist, "cuda")
    assert prob.status() == 0, "device status flagged during the timed steps"
    ms_per_step = total_ms / args.steps
    value = job_tflops(world, flops, ms_per_step)
    main_mean = statistics.mean(main_ms)

    # ---- warm L2: the same call back to back, no flush in between (context beside the flushed figure) ----
    warm_steps = max(1, min(args.steps, 50))
    w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    prob.step(0, stream)
    w0.record(stream)
    for _ in range(warm_steps):
        prob.step(0, stream)
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
        prob.step(0, stream)
        for dst, src in zip(host_out, outputs):
            dst.copy_(src, non_blocking=True)
        a1.record(stream)
        a1.synchronize()
        e2e_ms.append(a0.elapsed_time(a1))
        flush.fill_(1)
    e2e_val = job_tflops(world, flops, statistics.mean(e2e_ms))
    pipe_ms = e2e_pipelined(prob, max(4, e2e_steps))
    assert prob.status(0) == 0 and prob.status(1) == 0, "device status flagged during the end-to-end steps"
    del prob
    torch.cuda.empty_cache()

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
                       "N(0,1) seeded; O and softmax stats from the library sparse forward",
                       parallelism=(f"data-parallel shards x{world}: global problem of {world} x the "
                                    "workload's sequences, each rank its own (sequence, kv head) units, "
                                    "no collective on the data path") if world > 1 else "single GPU"),
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": tag, "kernel_ms": main_mean,
                     "peak_source": f"{pk_src} bf16_tflops (burst; fp16 has the same dense rate)",
                     "whole_call_frac": value / world / peak},
        "e2e": {"value": e2e_val, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": statistics.mean(e2e_ms),
                "pipelined": {"value": job_tflops(world, flops, pipe_ms), "unit": "TFLOP/s", "ms_per_step": pipe_ms,
                              "how": "two device buffer sets; copy in, call, copy out on three streams, overlapped"}},
        "warm_l2": {"value": job_tflops(world, flops, warm_ms), "unit": "TFLOP/s", "ms_per_step": warm_ms,
                    "steps": warm_steps},
        "gpu_launches": launches_per_step * args.steps,  # of the timed (whole-call) pass
        "clocks": clocks.summary(),
        "wall_s_timed_region": t_wall,
    }
    if nsa:
        line["roofline"]["useful_flops_frac"] = achieved * nsa_useful_flops(p) / flops / peak
    if world == 1 and not args.no_extra_workloads:
        line["workloads"] = extra_workloads(args, flush, stream, lib, peak)
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


def extra_workloads(args, flush, stream, lib, peak, steps=10, warmup=3):
    """The other workloads beside the headline one: per workload and dQ mode, the whole call and the
    main kernel (mean ms over `steps` flushed steps) and their fractions of the tensor peak."""
    import torch
    out = {}
    # dQ modes: False atomic, True split partial buffers (NSA: per-slot partials), 2 ordered single buffer
    for idx, det in ((2, False), (2, True), (2, 2), (3, False), (3, 2), (4, False), (4, True), (4, 2)):
        if idx == args.workload and det is False:
            continue
        p, flops, cfg = workload_info(idx)
        prob = Problem(p, det)
        for _ in range(warmup):
            prob.step(0, stream)
            flush.fill_(1)
        call_ms, main_ms = time_calls(prob, steps, flush, stream, lib)
        ok = prob.status() == 0
        call, main = statistics.mean(call_ms), statistics.mean(main_ms)
        mode = {False: "atomic", True: "split", 2: "ordered"}[det]
        entry = {"workload": cfg["workload"], "dq_mode": mode, "call_ms": call, "main_kernel_ms": main,
                 "tflops": flops / (call * 1e-3) / 1e12, "main_kernel_tflops": flops / (main * 1e-3) / 1e12,
                 "whole_call_frac": flops / (call * 1e-3) / 1e12 / peak,
                 "main_kernel_frac": flops / (main * 1e-3) / 1e12 / peak, "steps": steps, "device_status_clean": ok}
        if isinstance(p, synth.NsaProblem):
            uf = nsa_useful_flops(p)
            entry["useful_flops"] = uf
            entry["slot_flops"] = flops
            entry["main_kernel_useful_frac"] = uf / (main * 1e-3) / 1e12 / peak
        out[f"w{idx}" + {"atomic": "", "split": "_det", "ordered": "_ordered"}[mode]] = entry
        del prob
        torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=1, choices=[1, 2, 3, 4])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra-workloads", action="store_true",
                    help="time only the chosen workload (default: also workloads 2-4 in both dQ modes)")
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
