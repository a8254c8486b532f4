"""Benchmark of the document-masked core-attention hot path on GB300.

One step = one forward (ca_forward) + one backward (ca_backward) of the
rebatched CA-task pool over one synthetic 65536-token packed chunk shaped like
a Llama-3-8B layer (32 query / 8 KV heads, head_dim 128, documents with
lognormal lengths, median 2048, sigma 1.5, one CA-task per document; seed 0).
The metric counts 12 * head_dim * H_q FLOPs per causal (token, key) pair:
4 d forward and 8 d backward.

Printed (rank 0, one JSON line): whole-job TFLOP/s over the timed steps with
inputs resident in HBM (`value`), the same through the C ABI with host
buffers (`e2e`: pinned host -> device copies of Q, K, V, dO and device -> host
copies of O, LSE, dQ, dK, dV of every step inside the timed region, the copies
of the next and previous steps overlapping each step's compute on their own
streams; the one-stream serial schedule is reported beside it), the roofline
of the dominant kernel (the backward main kernel, timed live with CUDA events
on its stream), the clocks seen during the timed region, a sustained region of
at least 2.5 s of back-to-back steps with its clock samples binned by SM MHz
(`sustained`), the rebatched CA-task pool and the 512K long-context chunk
timed per launch (`more_configs`), and the fp64 oracle timed on the host cores
on a bounded sample of the same workload (`cpu_baseline`, with the full
chunk's time extrapolated from it and labelled as such).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

With --impl reference the oracle itself is the measured arm: each step runs
the oracle's forward + backward on a bounded sample (a prefix of the chunk's
documents) on the host cores.  Under torchrun (N > 1) every rank runs an
independent replica with its own seed (no data-path collective) and the
slowest rank's time is used.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
NOMINAL_DENSE_BF16_TFLOPS = 2250.0  # GB300 nominal dense bf16 (without 2:4 sparsity)
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "core-attention fwd+bwd TFLOP/s (causal-pair FLOPs), % of GB300 BF16 tensor peak"
UNIT = "TFLOP/s"
FALLBACK = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK), "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 50 ms in a thread;
    the summary keeps the samples read between mark_start() and mark_end()."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None
        self.thread = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.rows.append((time.time(), parts))

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0=None, t1=None, bins=False):
        """Median / min SM clock, max power and the throttle reasons seen in
        [t0, t1] (default: the marked region); with bins, the sample count per
        30 MHz bin of SM clock."""
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        t0 = self.t0 if t0 is None else t0
        t1 = self.t1 if t1 is None else t1
        rows = [r for t, r in self.rows if t0 is None or t1 is None or t0 <= t <= t1 + 0.05]
        if not rows:
            rows = [r for _, r in self.rows]
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        pw = [num(r[3]) for r in rows if num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        out = {"sm_mhz": statistics.median(sm) if sm else None, "sm_mhz_min": min(sm) if sm else None,
               "sm_max_mhz": max(mx) if mx else None, "power_w_max": max(pw) if pw else None,
               "reasons": sorted(reasons), "samples": len(rows)}
        if bins:
            hist = {}
            for x in sm:
                b = int(x // 30 * 30)
                hist[f"{b}-{b + 29}"] = hist.get(f"{b}-{b + 29}", 0) + 1
            out["sm_mhz_bins"] = dict(sorted(hist.items()))
        return out


def measured_traffic(kernel_file="traffic_bwd_main_llama8b_chunk_64k.json"):
    """DRAM bytes per launch of one kernel from its committed ncu summary
    (default: the backward main kernel), or None when the kernel's sources
    have changed since the capture (their hash differs) or no summary
    exists."""
    import hashlib
    path = os.path.join(ROOT, "profiles", kernel_file)
    try:
        with open(path) as f:
            d = json.load(f)
        h = hashlib.sha256()
        for src in d["sources"]:
            with open(os.path.join(ROOT, src), "rb") as f:
                h.update(f.read())
        if h.hexdigest() != d["sources_sha256"]:
            return None
        return int(d["dram_read_bytes"]) + int(d["dram_write_bytes"])
    except (OSError, KeyError, ValueError):
        return None


def dist_setup(n_gpus):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl"
        try:
            import torch
            if not torch.cuda.is_available():
                backend = "gloo"
        except Exception:
            backend = "gloo"
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- oracle sample

def oracle_sample_workload(w, pair_budget: int, kv_groups: int = 1):
    """Bounded sample of the chunk: its leading documents whose causal pairs
    per head stay within pair_budget (or the leading tokens of the first one),
    each one CA-task, with the first ``kv_groups`` KV heads and their query
    heads."""
    import workloads as W
    lens = []
    acc = 0
    for L in w.doc_len:
        p = int(L) * (int(L) + 1) // 2
        if acc + p > pair_budget:
            if not lens:  # the first document alone is over budget: keep its leading tokens
                l = int((2 * pair_budget) ** 0.5)
                while l > 1 and l * (l + 1) // 2 > pair_budget:
                    l -= 1
                lens.append(max(1, l))
            break
        lens.append(int(L))
        acc += p
    G = w.num_q_heads // w.num_kv_heads
    return W.custom(f"{w.name}_prefix{len(lens)}_kv{kv_groups}", lens,
                    [(i, 0, l, 0, l) for i, l in enumerate(lens)], G * kv_groups, kv_groups, w.head_dim,
                    seed=w.seed)


def time_oracle(ws, steps: int):
    """Full fp64 oracle forward + backward on the sample workload, `steps`
    times; returns (seconds per step, counted FLOPs per step)."""
    import oracle
    import workloads as W
    q, k, v, do = W.make_tensors(ws, device="cpu")
    pb = oracle.Problem(ws, q, k, v, do)
    f, b = oracle.flops(ws)
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        oracle.forward(pb)
        oracle.backward(pb)
        times.append(time.perf_counter() - t0)
    return float(np.mean(times)), f + b


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def run_reference(args, rank, world):
    import oracle
    import workloads as W
    if rank != 0:
        return
    w = W.llama8b_chunk(seed=0)
    ws = oracle_sample_workload(w, args.oracle_pairs // 4)
    oracle.build()
    t_warm, _ = time_oracle(ws, max(1, min(args.warmup, 1)))
    t, flops = time_oracle(ws, args.steps)
    value = flops / t / 1e12
    sample = (f"{ws.n_docs} leading documents ({ws.total_q} tokens, {int(oracle.task_pairs(ws).sum())} causal "
              f"pairs/head) of the chunk, {ws.num_q_heads} query heads sharing {ws.num_kv_heads} KV head(s), "
              f"full fp64 forward + backward per step")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "seed": 0, "sample": ws.name},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def measure_e2e(args, plan, stream, inputs, fwd_out, grads, ws, world, flops_step, step_ms):
    """The same step through the C ABI with host buffers: pinned host -> device
    copies of Q, K, V, dO and device -> host copies of O, LSE, dQ, dK, dV inside
    the timed region, every step.

    Two schedules over the same host buffers.  Serial: one stream runs each
    step's copies in, forward, backward and copies out in turn.  Overlapped (the
    reported value): device inputs and outputs are double-buffered, the
    host -> device copies run on their own stream and the device -> host copies on
    another, so step k+1's inputs arrive and step k-1's gradients leave while step
    k computes (events keep each buffer slot from being reused early); the timed
    region starts before the first copy in and ends after the last copy out."""
    import torch
    q, k, v, do = inputs
    o, lse = fwd_out
    dq, dk, dv = grads
    sh = stream.cuda_stream
    hq = q.cpu().pin_memory()
    hk = k.cpu().pin_memory()
    hv = v.cpu().pin_memory()
    hdo = do.cpu().pin_memory()
    h_out = tuple(torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in (o, lse, dq, dk, dv))
    h_in = (hq, hk, hv, hdo)
    h2d = sum(x.numel() * x.element_size() for x in h_in)
    d2h = sum(x.numel() * x.element_size() for x in h_out)
    dev_in = [tuple(torch.empty_like(x) for x in (q, k, v, do)) for _ in range(2)]
    # every slot has its own O and LSE: the forward's results leave the device too
    dev_out = [tuple(torch.empty_like(x) for x in (o, lse, dq, dk, dv)) for _ in range(2)]

    def compute(slot):
        qi, ki, vi, doi = dev_in[slot]
        oo, lo, dqo, dko, dvo = dev_out[slot]
        plan.forward(qi, ki, vi, oo, lo, ws, stream=sh)
        plan.backward(qi, ki, vi, oo, lo, doi, dqo, dko, dvo, ws, stream=sh)

    def serial_step():
        with torch.cuda.stream(stream):
            for dst, src in zip(dev_in[0], h_in):
                dst.copy_(src, non_blocking=True)
            compute(0)
            for dst, src in zip(h_out, dev_out[0]):
                dst.copy_(src, non_blocking=True)

    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]    # inputs of the slot are on the device
    ev_done = [torch.cuda.Event() for _ in range(2)]  # the slot's step computed (inputs free, outputs ready)
    ev_out = [torch.cuda.Event() for _ in range(2)]   # the slot's outputs reached the host (outputs free)

    def overlapped(n):
        used = [False, False]
        last = 0
        for i in range(n):
            slot = i % 2
            with torch.cuda.stream(s_in):
                if used[slot]:
                    s_in.wait_event(ev_done[slot])
                for dst, src in zip(dev_in[slot], h_in):
                    dst.copy_(src, non_blocking=True)
                ev_in[slot].record(s_in)
            stream.wait_event(ev_in[slot])
            if used[slot]:
                stream.wait_event(ev_out[slot])
            with torch.cuda.stream(stream):
                compute(slot)
            ev_done[slot].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[slot])
                for dst, src in zip(h_out, dev_out[slot]):
                    dst.copy_(src, non_blocking=True)
                ev_out[slot].record(s_out)
            used[slot] = True
            last = slot
        stream.wait_event(ev_out[last])  # the last copy out ends the region

    def timed(run):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        s_in.wait_event(start)
        s_out.wait_event(start)
        run()
        end.record(stream)
        stream.synchronize()
        torch.cuda.synchronize()
        return start.elapsed_time(end)

    warm = max(1, args.warmup // 2)
    # the overlapped region holds one pipeline fill (the first copy in) and one drain (the last copy
    # out), about 13 ms together; a training loop pays them once, so the region runs as long as the
    # sustained region (at least 60 steps)
    n_e2e = max(args.steps, 60, int(np.ceil(args.sustained_s * 1e3 / step_ms)))
    timed(lambda: [serial_step() for _ in range(warm)])
    barrier(world)
    serial_ms = max_over_ranks(timed(lambda: [serial_step() for _ in range(args.steps)]) / args.steps, world)
    timed(lambda: overlapped(warm))
    barrier(world)
    e2e_ms = max_over_ranks(timed(lambda: overlapped(n_e2e)) / n_e2e, world)
    if plan.device_status(stream=sh) != 0:
        raise RuntimeError("device error in the end-to-end region")
    return {"value": flops_step * world / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
            "copies": "in: Q, K, V, dO; out: O, LSE, dQ, dK, dV (pinned host buffers)",
            "steps": n_e2e, "serial_steps": args.steps,
            "schedule": "double-buffered: copies in of step k+1 and out of step k-1 on their own streams "
                        "during step k's compute",
            "serial_ms_per_step": serial_ms,
            "serial_value": flops_step * world / (serial_ms * 1e-3) / 1e12}


def measure_pair_backward(plan, stream, inputs, fwd_out, grads, ws, info, steps=4):
    """The backward main kernel on CTA pairs (CA_BWD_KERNEL_PAIR) against the
    default one-CTA kernel, each timed by the library's own events around the
    main launch, alternating; the plan is left on its default afterwards."""
    import torch

    from document_masked_core_gb300 import capi
    q, k, v, do = inputs
    o, lse = fwd_out
    dq, dk, dv = grads
    sh = stream.cuda_stream
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    for e in ev:
        e.record(stream)
    t = {capi.CA_BWD_KERNEL_SINGLE: [], capi.CA_BWD_KERNEL_PAIR: []}
    for r in range(2 * steps + 2):
        kind = (capi.CA_BWD_KERNEL_SINGLE, capi.CA_BWD_KERNEL_PAIR)[r % 2]
        plan.set_backward_kernel(kind)
        plan.set_timing_events(ev)
        with torch.cuda.stream(stream):
            plan.backward(q, k, v, o, lse, do, dq, dk, dv, ws, stream=sh)
        stream.synchronize()
        plan.set_timing_events(None)
        if r >= 2:  # the first of each is a warm-up
            t[kind].append(ev[3].elapsed_time(ev[4]))
    plan.set_backward_kernel(capi.CA_BWD_KERNEL_AUTO)
    if plan.device_status(stream=sh) != 0:
        raise RuntimeError("device error in the pair-kernel comparison")
    single = float(np.median(t[capi.CA_BWD_KERNEL_SINGLE]))
    pair = float(np.median(t[capi.CA_BWD_KERNEL_PAIR]))
    return {"single_main_ms": single, "pair_main_ms": pair,
            "single_main_tflops": info["flops_bwd"] / (single * 1e-3) / 1e12,
            "pair_main_tflops": info["flops_bwd"] / (pair * 1e-3) / 1e12,
            "note": "opt-in kernel (ca_plan_set_backward_kernel), not the default; same work, same counted FLOPs"}


def measure_masks(args, dev, stream, causal_pairs):
    """The sparse mask families on the same 64K lognormal chunk (lambda: sink
    64 + window 4096; causal blockwise: 256-token blocks, 1 sink block, 2
    window blocks; and a 64K pool of shared-question documents): fwd+bwd
    TFLOP/s over the visible pairs (12 d H_q per pair), and the density
    relative to the causal chunk."""
    import torch

    import document_masked_core_gb300 as ca
    import workloads as W

    out = {}
    for name, gen in W.MASKED_WORKLOADS.items():
        w = gen(seed=args.seed)
        q, k, v, do = W.make_tensors(w, device=dev)
        plan = ca.Plan.from_workload(w, stream=stream)
        info = plan.info()
        ws = torch.empty(max(16, info["workspace_bytes"]), dtype=torch.uint8, device=dev)
        o, lse = ca.alloc_forward(plan, device=dev)
        dq, dk, dv = ca.alloc_backward(plan, device=dev)
        sh = stream.cuda_stream
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]

        def step():
            plan.forward(q, k, v, o, lse, ws, stream=sh)
            ev[1].record(stream)
            plan.backward(q, k, v, o, lse, do, dq, dk, dv, ws, stream=sh)

        for _ in range(args.warmup):
            step()
        stream.synchronize()
        fwd, tot = [], []
        for _ in range(max(3, args.steps // 4)):
            ev[0].record(stream)
            step()
            ev[2].record(stream)
            stream.synchronize()
            fwd.append(ev[0].elapsed_time(ev[1]))
            tot.append(ev[0].elapsed_time(ev[2]))
        if plan.device_status(stream=sh) != 0:
            raise RuntimeError(f"device error in the {name} mask measurement")
        f_ms, t_ms = float(np.median(fwd)), float(np.median(tot))
        pairs = info["causal_pairs"]
        out[name] = {"workload": w.name, "visible_pairs_per_head": pairs,
                     "density_vs_causal_chunk": pairs / causal_pairs if name != "shared_question" else None,
                     "fwd_bwd_ms": t_ms, "forward_ms": f_ms,
                     "tflops": (info["flops_fwd"] + info["flops_bwd"]) / (t_ms * 1e-3) / 1e12,
                     "forward_tflops": info["flops_fwd"] / (f_ms * 1e-3) / 1e12}
        plan.close()
        del q, k, v, do, o, lse, dq, dk, dv, ws
    return out


def measure_decode(args, dev, stream, pk):
    """Decode shape (one new token per sequence against 131072 cached tokens,
    16 sequences, 32 q / 8 kv heads): forward time with the in-launch
    split-KV (automatic) and without it, against the HBM roofline
    (algorithmic bytes: every K and V row of every sequence read once, Q, O
    and LSE once)."""
    import torch

    import document_masked_core_gb300 as ca
    import workloads as W

    w = W.decode_batch(seed=args.seed, n_seq=16, context=131072, q_len=1)
    q, k, v, _ = W.make_tensors(w, device=dev, need_grad_inputs=False)
    hbm = float(pk.get("hbm_gbs", FALLBACK["hbm_gbs"]))
    nbytes = int(w.doc_len.sum()) * w.num_kv_heads * w.head_dim * 2 * 2 + w.total_q * w.num_q_heads * (
        w.head_dim * 2 * 2 + 4)
    out = {"workload": w.name, "algorithmic_bytes": nbytes}
    for mode, split in (("split", 0), ("unsplit", -1)):
        plan = ca.Plan.from_workload(w, stream=stream)
        plan.set_kv_split(split)
        info = plan.info()
        ws = torch.empty(max(16, info["workspace_bytes"]), dtype=torch.uint8, device=dev)
        o, lse = ca.alloc_forward(plan, device=dev)
        sh = stream.cuda_stream
        for _ in range(args.warmup):
            plan.forward(q, k, v, o, lse, ws, stream=sh)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n = max(5, args.steps // 4)
        e0.record(stream)
        for _ in range(n):
            plan.forward(q, k, v, o, lse, ws, stream=sh)
        e1.record(stream)
        stream.synchronize()
        if plan.device_status(stream=sh) != 0:
            raise RuntimeError("device error in the decode measurement")
        ms = e0.elapsed_time(e1) / n
        gbs = nbytes / (ms * 1e-3) / 1e9
        out[mode] = {"forward_ms": ms, "items": info["n_fwd_items"],
                     "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm}}
        plan.close()
    return out


def measure_split_kv(args, dev, stream, pk):
    """Partial prefill with split KV: 4096 new tokens at positions
    131072..135167, the 135168-key context cut into 8 contiguous blocks, one
    CA-task per block (float32 partial O, LSE), then ca_merge.  Reports the
    forward over the blocks (TFLOP/s, 4 d FLOPs per causal pair per query
    head) and the merge against the measured HBM bandwidth (algorithmic bytes:
    every partial O and LSE read once, O (bf16) and LSE written once)."""
    import torch

    import document_masked_core_gb300 as ca
    import workloads as W

    wsplit = W.split_kv_prefill(seed=args.seed)
    whole = W.split_kv_prefill(seed=args.seed, split=False)
    nb = wsplit.n_tasks
    q, k, v, _ = W.make_tensors(whole, device=dev, need_grad_inputs=False)
    nq, hq, d = q.shape
    q8 = q.repeat(nb, 1, 1)  # the blocks share the query rows; tasks are packed one after another
    plan = ca.Plan.from_workload(wsplit, o_dtype=ca.CA_DTYPE_FP32, stream=stream)
    info = plan.info()
    ws = torch.empty(max(16, info["workspace_bytes"]), dtype=torch.uint8, device=dev)
    o_p, lse_p = ca.alloc_forward(plan, device=dev)
    o = torch.empty((nq, hq, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((nq, hq), dtype=torch.float32, device=dev)
    parts_o = [o_p[b * nq:(b + 1) * nq] for b in range(nb)]
    parts_l = [lse_p[b * nq:(b + 1) * nq] for b in range(nb)]
    sh = stream.cuda_stream
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]

    def step():
        plan.forward(q8, k, v, o_p, lse_p, ws, stream=sh)
        ev[1].record(stream)
        ca.merge(parts_o, parts_l, nq, hq, d, o, lse, parts_dtype=ca.CA_DTYPE_FP32,
                 out_dtype=ca.CA_DTYPE_BF16, stream=sh)

    for _ in range(args.warmup):
        step()
    stream.synchronize()
    fwd_ms, merge_ms = [], []
    for _ in range(args.steps):
        ev[0].record(stream)
        step()
        ev[2].record(stream)
        stream.synchronize()
        fwd_ms.append(ev[0].elapsed_time(ev[1]))
        merge_ms.append(ev[1].elapsed_time(ev[2]))
    if plan.device_status(stream=sh) != 0:
        raise RuntimeError("device error in the split-KV measurement")
    f_ms, m_ms = float(np.median(fwd_ms)), float(np.median(merge_ms))
    merge_bytes = nb * nq * hq * (d * 4 + 4) + nq * hq * (d * 2 + 4)
    hbm = float(pk.get("hbm_gbs", FALLBACK["hbm_gbs"]))
    gbs = merge_bytes / (m_ms * 1e-3) / 1e9
    out = {
        "workload": wsplit.name, "blocks": nb, "forward_ms": f_ms, "merge_ms": m_ms,
        "forward_tflops": info["flops_fwd"] / (f_ms * 1e-3) / 1e12,
        "forward_plus_merge_tflops": info["flops_fwd"] / ((f_ms + m_ms) * 1e-3) / 1e12,
        "merge_roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                           "traffic": None, "algorithmic_bytes": merge_bytes},
    }
    plan.close()
    return out


def measure_config(args, dev, stream, pk, name, steps):
    """One more configuration of the same kernels, fwd+bwd: the rebatched
    CA-task pool (131072 query tokens of token-granular shards of 16 documents
    of 8K..128K tokens, 32 q / 8 kv heads) or the 512K long-context chunk (one
    262144-token document plus lognormal documents, 64 q / 8 kv heads).  Per
    launch CUDA events on the launching stream; TFLOP/s over counted causal
    pairs (4 d forward, 8 d backward per pair per query head)."""
    import torch

    import document_masked_core_gb300 as ca
    import workloads as W

    w = W.WORKLOADS[name](seed=args.seed)
    q, k, v, do = W.make_tensors(w, device=dev)
    plan = ca.Plan.from_workload(w, stream=stream)
    info = plan.info()
    ws = torch.empty(max(16, info["workspace_bytes"]), dtype=torch.uint8, device=dev)
    o, lse = ca.alloc_forward(plan, device=dev)
    dq, dk, dv = ca.alloc_backward(plan, device=dev)
    sh = stream.cuda_stream
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(steps)]
    for row in ev:  # torch creates the underlying cudaEvent on first record
        for e in row:
            e.record(stream)

    def step():
        plan.forward(q, k, v, o, lse, ws, stream=sh)
        plan.backward(q, k, v, o, lse, do, dq, dk, dv, ws, stream=sh)

    for _ in range(3):
        step()
    stream.synchronize()
    t0 = time.time()
    for s in range(steps):
        plan.set_timing_events(ev[s])
        step()
    stream.synchronize()
    t1 = time.time()
    plan.set_timing_events(None)
    if plan.device_status(stream=sh) != 0:
        raise RuntimeError(f"device error in the {name} measurement")
    f_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in ev]))
    b_ms = float(np.mean([e[2].elapsed_time(e[5]) for e in ev]))
    m_ms = float(np.mean([e[3].elapsed_time(e[4]) for e in ev]))
    peak = float(pk.get("bf16_tflops", FALLBACK["bf16_tflops"]))
    ff, fb = info["flops_fwd"], info["flops_bwd"]
    out = {"workload": w.name, "tokens": w.total_q, "documents": w.n_docs, "tasks": w.n_tasks,
           "heads": f"{w.num_q_heads}q/{w.num_kv_heads}kv", "causal_pairs_per_head": info["causal_pairs"],
           "steps": steps, "warmup": 3, "forward_ms": f_ms, "backward_ms": b_ms, "bwd_main_ms": m_ms,
           "forward_tflops": ff / (f_ms * 1e-3) / 1e12, "backward_tflops": fb / (b_ms * 1e-3) / 1e12,
           "fwd_bwd_tflops": (ff + fb) / ((f_ms + b_ms) * 1e-3) / 1e12,
           "pct_of_burst_peak": 100.0 * (ff + fb) / ((f_ms + b_ms) * 1e-3) / 1e12 / peak,
           "roofline": {"kernel": "ca_bwd_main_kernel", "bound": "tensor", "unit": "TFLOP/s", "peak": peak,
                        "achieved": fb / (m_ms * 1e-3) / 1e12, "frac": fb / (m_ms * 1e-3) / 1e12 / peak},
           "forward_roofline": {"kernel": "ca_fwd_kernel", "bound": "tensor", "unit": "TFLOP/s", "peak": peak,
                                "achieved": ff / (f_ms * 1e-3) / 1e12, "frac": ff / (f_ms * 1e-3) / 1e12 / peak},
           "window": (t0, t1)}
    plan.close()
    del q, k, v, do, o, lse, dq, dk, dv, ws
    torch.cuda.empty_cache()
    return out


def measure_tiny(args, dev, stream):
    """The tiny packed chunk (2048 tokens, documents of 1024, 512, 256 and 256
    tokens, 4 q / 1 kv head, head_dim 64), which is launch-latency bound:
    fwd+bwd per step issued call by call against the same two calls captured
    once into a CUDA graph and replayed (both timed over back-to-back steps
    with CUDA events)."""
    import torch

    import document_masked_core_gb300 as ca
    import workloads as W

    w = W.tiny_chunk(seed=args.seed)
    q, k, v, do = W.make_tensors(w, device=dev)
    plan = ca.Plan.from_workload(w, stream=stream)
    info = plan.info()
    ws = torch.empty(max(16, info["workspace_bytes"]), dtype=torch.uint8, device=dev)
    o, lse = ca.alloc_forward(plan, device=dev)
    dq, dk, dv = ca.alloc_backward(plan, device=dev)
    sh = stream.cuda_stream

    def step():
        plan.forward(q, k, v, o, lse, ws, stream=sh)
        plan.backward(q, k, v, o, lse, do, dq, dk, dv, ws, stream=sh)

    n = 200
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            step()
        e1.record(stream)
    stream.synchronize()
    eager_ms = e0.elapsed_time(e1) / n
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        plan.forward(q, k, v, o, lse, ws)
        plan.backward(q, k, v, o, lse, do, dq, dk, dv, ws)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            g.replay()
        e0.record(stream)
        for _ in range(n):
            g.replay()
        e1.record(stream)
    stream.synchronize()
    graph_ms = e0.elapsed_time(e1) / n
    if plan.device_status(stream=sh) != 0:
        raise RuntimeError("device error in the tiny-chunk measurement")
    fl = info["flops_fwd"] + info["flops_bwd"]
    out = {"workload": w.name, "steps": n, "eager_ms": eager_ms, "graph_ms": graph_ms,
           "eager_tflops": fl / (eager_ms * 1e-3) / 1e12, "graph_tflops": fl / (graph_ms * 1e-3) / 1e12,
           "bound": "launch latency (4 kernels and a memset per step)"}
    plan.close()
    return out


# ----------------------------------------------------------------------------- GPU arm

def run_gpu(args, rank, world, local):
    import torch

    import document_masked_core_gb300 as ca
    import workloads as W

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    seed = args.seed + rank
    w = W.llama8b_chunk(seed=seed, total=args.tokens)
    q, k, v, do = W.make_tensors(w, device=dev)
    stream = torch.cuda.Stream(device=dev)
    t0 = time.perf_counter()
    plan = ca.Plan.from_workload(w, stream=stream)
    plan_ms = (time.perf_counter() - t0) * 1e3
    plan.set_backward_kernel({"auto": 0, "single": 1, "pair": 2}[args.backward_kernel])
    info = plan.info()
    ws = torch.empty(max(16, info["workspace_bytes"]), dtype=torch.uint8, device=dev)
    o, lse = ca.alloc_forward(plan, device=dev)
    dq, dk, dv = ca.alloc_backward(plan, device=dev)
    flops_step = info["flops_fwd"] + info["flops_bwd"]
    sh = stream.cuda_stream

    def step():
        plan.forward(q, k, v, o, lse, ws, stream=sh)
        plan.backward(q, k, v, o, lse, do, dq, dk, dv, ws, stream=sh)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    stream.synchronize()
    if plan.device_status(stream=sh) != 0:
        raise RuntimeError("device error during warm-up")

    # ---- timed region: inputs resident in HBM (Q, dO 512 MiB, K, V 128 MiB each: larger than L2)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    for row in ev:  # torch creates the underlying cudaEvent on first record
        for e in row:
            e.record(stream)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local if "CUDA_VISIBLE_DEVICES" not in os.environ else 0)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    clocks.mark_start()
    with torch.cuda.stream(stream):
        start.record(stream)
        for s in range(args.steps):
            plan.set_timing_events(ev[s])
            step()
        end.record(stream)
    stream.synchronize()
    clocks.mark_end()
    plan.set_timing_events(None)
    torch.cuda.synchronize()
    barrier(world)
    if plan.device_status(stream=sh) != 0:
        raise RuntimeError("device error in the timed region")
    ms_local = start.elapsed_time(end) / args.steps
    ms = max_over_ranks(ms_local, world)

    # ---- a sustained region of at least 2 s of back-to-back steps (the clock
    # under a long load settles below its burst value; samples binned by MHz)
    sustained = None
    if not args.no_sustained:
        n_sus = max(args.steps, int(np.ceil(args.sustained_s * 1e3 / ms_local)))
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        w0 = time.time()
        with torch.cuda.stream(stream):
            s0.record(stream)
            for _ in range(n_sus):
                step()
            s1.record(stream)
        stream.synchronize()
        w1 = time.time()
        barrier(world)
        if plan.device_status(stream=sh) != 0:
            raise RuntimeError("device error in the sustained region")
        sus_ms = max_over_ranks(s0.elapsed_time(s1) / n_sus, world)
        sustained = {"steps": n_sus, "seconds": sus_ms * n_sus * 1e-3, "ms_per_step": sus_ms,
                     "value": flops_step * world / (sus_ms * 1e-3) / 1e12, "unit": UNIT,
                     "window": (w0, w1)}
    value = flops_step * world / (ms * 1e-3) / 1e12
    fwd_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in ev]))
    pre_ms = float(np.mean([e[2].elapsed_time(e[3]) for e in ev]))
    main_ms = float(np.mean([e[3].elapsed_time(e[4]) for e in ev]))
    fin_ms = float(np.mean([e[4].elapsed_time(e[5]) for e in ev]))

    # ---- end to end through the C ABI with host buffers
    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(args, plan, stream, (q, k, v, do), (o, lse), (dq, dk, dv), ws, world, flops_step,
                          ms_local)

    # the opt-in CTA-pair backward main kernel on the same chunk, for comparison (not the headline)
    pair = None
    if not args.no_more_configs and w.head_dim == 128:
        pair = measure_pair_backward(plan, stream, (q, k, v, do), (o, lse), (dq, dk, dv), ws, info)
        plan.set_backward_kernel({"auto": 0, "single": 1, "pair": 2}[args.backward_kernel])

    pk, pk_kind = peaks()
    split_kv = None
    if not args.no_split_kv:
        split_kv = measure_split_kv(args, dev, stream, pk)
    masks = None
    if not args.no_masks:
        masks = measure_masks(args, dev, stream, info["causal_pairs"])
    decode = None
    if not args.no_decode:
        decode = measure_decode(args, dev, stream, pk)
    more = {}
    if not args.no_more_configs:
        more["tiny_chunk"] = measure_tiny(args, dev, stream)
        more["rebatched_pool"] = measure_config(args, dev, stream, pk, "pool", steps=8)
        more["long_context_chunk"] = measure_config(args, dev, stream, pk, "long", steps=3)
    peak = float(pk.get("bf16_tflops", FALLBACK["bf16_tflops"]))
    peak_sus = float(pk.get("bf16_tflops_sustained", FALLBACK["bf16_tflops_sustained"]))
    main_tf = info["flops_bwd"] / (main_ms * 1e-3) / 1e12

    clocks.stop()
    if sustained is not None:
        w0, w1 = sustained.pop("window")
        sustained["clocks"] = clocks.summary(w0, w1, bins=True)
        c = sustained["clocks"]
        if c["sm_mhz"] and c["sm_max_mhz"]:
            # time x median clock: what the same work takes at the maximum clock if it scales with the clock
            sustained["ms_per_step_at_max_clock_est"] = sustained["ms_per_step"] * c["sm_mhz"] / c["sm_max_mhz"]
    for name, m in more.items():
        if "window" in m:
            w0, w1 = m.pop("window")
            m["clocks"] = clocks.summary(w0, w1)

    line = None
    if rank == 0:
        # CPU baseline: the oracle on a bounded sample of the same workload
        cpu = None
        if not args.no_cpu_baseline:
            import oracle
            oracle.build()
            wsamp = oracle_sample_workload(w, args.oracle_pairs, kv_groups=2)
            t_cpu, f_cpu = time_oracle(wsamp, 1)
            cpu = {"value": f_cpu / t_cpu / 1e12, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                   "sample": (f"{wsamp.n_docs} leading documents ({wsamp.total_q} tokens, "
                              f"{int(oracle.task_pairs(wsamp).sum())} causal pairs/head) of the chunk, "
                              f"{wsamp.num_q_heads} query heads sharing {wsamp.num_kv_heads} KV head(s), full "
                              f"fp64 forward + backward; {t_cpu:.1f} s")}
            cpu["extrapolated_full_s"] = flops_step / (cpu["value"] * 1e12)
            cpu["extrapolation"] = ("extrapolation, not a measurement: the full chunk's counted FLOPs per step "
                                    "divided by the sample's measured CPU rate")
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {
                "workload": w.name, "seed": seed, "tokens": w.total_q, "documents": w.n_docs,
                "heads": f"{w.num_q_heads}q/{w.num_kv_heads}kv", "head_dim": w.head_dim,
                "causal_pairs_per_head": info["causal_pairs"], "flops_per_step": flops_step,
                "flop_count": "12*head_dim*H_q*causal_pairs (4d forward + 8d backward)",
                "l2": (f"inputs larger than L2 (Q and dO {q.numel() * 2 >> 20} MiB, K and V "
                       f"{k.numel() * 2 >> 20} MiB each; L2 is 129 MB)"),
                "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                "backward_kernel": args.backward_kernel,
                "plan_ms": plan_ms,
            },
            "pct_of_peak": {"burst": 100.0 * value / world / peak, "sustained": 100.0 * value / world / peak_sus,
                            "peaks": pk_kind,
                            "nominal_dense": 100.0 * value / world / NOMINAL_DENSE_BF16_TFLOPS,
                            "nominal_note": "vs the nominal 2.25 PFLOP/s dense bf16 of a GB300 (context only)"},
            "tflops_14d_convention": {"value": value * 14.0 / 12.0,
                                      "note": "FlashAttention's 2.5x backward convention (14 d per pair); "
                                              "not the headline, which counts 12 d"},
            "parts_ms": {"forward": fwd_ms, "bwd_preprocess": pre_ms, "bwd_main": main_ms,
                         "bwd_dq_finalize": fin_ms},
            "parts_tflops": {"forward": info["flops_fwd"] / (fwd_ms * 1e-3) / 1e12,
                             "backward": info["flops_bwd"] / ((pre_ms + main_ms + fin_ms) * 1e-3) / 1e12},
            "roofline": {"kernel": "ca_bwd_pair_kernel" if args.backward_kernel == "pair" else "ca_bwd_main_kernel",
                         "bound": "tensor", "achieved": main_tf, "peak": peak,
                         "unit": "TFLOP/s", "frac": main_tf / peak,
                         "traffic": None if args.backward_kernel == "pair" else measured_traffic(),
                         "traffic_unit": "bytes per launch (ncu dram read + write, profiles/)",
                         "peak_kind": f"bf16 burst, {pk_kind}",
                         "algorithmic": "8*head_dim*H_q*causal_pairs per launch"},
            "forward_roofline": {"kernel": "ca_fwd_kernel", "bound": "tensor",
                                 "achieved": info["flops_fwd"] / (fwd_ms * 1e-3) / 1e12, "peak": peak,
                                 "unit": "TFLOP/s", "frac": info["flops_fwd"] / (fwd_ms * 1e-3) / 1e12 / peak,
                                 "traffic": measured_traffic("traffic_fwd_llama8b_chunk_64k.json"),
                                 "traffic_unit": "bytes per launch (ncu dram read + write, profiles/)",
                                 "algorithmic": "4*head_dim*H_q*causal_pairs per launch; algorithmic bytes "
                                                "Q, K, V, O, LSE once = 1.30 GB"},
            "e2e": e2e,
            "split_kv_prefill": split_kv,
            "sparse_masks": masks,
            "decode": decode,
            "sustained": sustained,
            "more_configs": more or None,
            "backward_pair_kernel": pair,
            "gpu_launches": 4 * args.steps,
            "clocks": clocks.summary(),
            "cpu_baseline": cpu,
        }
    plan.close()
    return line


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--oracle-pairs", type=int, default=30_000_000,
                    help="causal pairs per head of the oracle's sample (bounds its CPU time)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end measurement")
    ap.add_argument("--no-split-kv", action="store_true", help="skip the split-KV prefill + merge measurement")
    ap.add_argument("--no-masks", action="store_true", help="skip the sparse-mask measurement")
    ap.add_argument("--no-decode", action="store_true", help="skip the decode (split-KV) measurement")
    ap.add_argument("--no-sustained", action="store_true", help="skip the sustained (>= 2 s) region")
    ap.add_argument("--sustained-s", type=float, default=2.5, help="length of the sustained region (seconds)")
    ap.add_argument("--no-more-configs", action="store_true",
                    help="skip the rebatched-pool and 512K-chunk measurements")
    ap.add_argument("--backward-kernel", choices=["auto", "single", "pair"], default="auto",
                    help="backward main kernel of the headline step (ca_plan_set_backward_kernel)")
    ap.add_argument("--tokens", type=int, default=65536,
                    help="chunk size (65536 = the measured workload; smaller sizes only for profiling captures)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        raise SystemExit("--warmup must be >= 3")
    rank, world, local = dist_setup(args.gpus)
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
            return
        from document_masked_core_gb300 import build
        if rank == 0:
            build.build()
        barrier(world)
        line = run_gpu(args, rank, world, local)
        if rank == 0 and line is not None:
            print(json.dumps(line), flush=True)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
