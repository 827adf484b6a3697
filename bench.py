#!/usr/bin/env python
"""Benchmark of the MSA training hot path (index top-k -> sparse forward -> fused backward).

One step = msa_index_topk + msa_sparse_fwd + msa_bwd over one batch of
synthetic inputs already resident in HBM. Default workload: B=1, T=131072,
Hq=32, G=8, d=128, d_idx=64, Bk=128, k=16. Prints ONE JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config ID] [--impl gb300|reference]

--impl reference times the fp64 CPU oracle (as it stands) on a bounded sample
of the same workload, per step, on the host cores.

Multi-GPU: launched with torch.distributed.run, one process per GPU; every rank
runs its own batch (the path shards over the batch with no collective:
weak scaling); a barrier brackets the timed region and rank 0 reports the
max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "MSA fwd+bwd tokens/s and achieved TFLOP/s vs GB300 BF16 peak (k=16, Bk=128)"


def n_selected(w) -> int:
    """Selected, causally visible (query, key) pairs per (b, g) when every
    query keeps min(k, visible) blocks: the own block's t-c*Bk+1 keys plus
    Bk keys for each of min(k-1, c) earlier blocks."""
    Bk = w.Bk
    tot = 0
    for c in range(w.n_blocks):
        tot += Bk * (Bk + 1) // 2 + Bk * Bk * min(c, w.k - 1)
    return tot


def counted_flops(w):
    """Counted FLOPs: full causal index branch + selected-block main fwd/bwd + KL bwd."""
    ns = n_selected(w) * w.B * w.G
    hg = w.Hq // w.G
    idx = w.d_idx * w.B * w.G * w.T * (w.T + 1)
    fwd = 4 * w.d * hg * ns
    bwd = 10 * w.d * hg * ns
    kl = 6 * w.d_idx * ns
    return dict(index=idx, fwd=fwd, bwd=bwd + kl, total=idx + fwd + bwd + kl)


def algorithmic_bytes(w) -> dict:
    """HBM bytes each entry point must move at least: every input read once and
    every output written once, in the library's storage types (bf16 inputs and
    O; int32 block_idx; fp32 LSE, KL and gradients)."""
    bt, hq, G, d, E, k = w.B * w.T, w.Hq, w.G, w.d, w.d_idx, w.k
    q = bt * hq * d * 2            # Q, dO, O (bf16)
    kv = bt * G * d * 2            # K, V (bf16)
    qi, ki = bt * G * E * 2, bt * E * 2
    bi = bt * G * k * 4
    lse = bt * hq * 4
    index = qi + ki + bi
    fwd = q + 2 * kv + bi + q + lse
    bwd = (q + 2 * kv + q + q + lse + qi + ki + bi     # Q, K, V, O, dO, LSE, q_idx, k_idx, block_idx
           + 2 * q + 2 * (2 * kv) + 2 * qi + 2 * ki + bt * G * 4)  # dQ, dK, dV, dq_idx, dk_idx (fp32), KL
    return dict(index=index, fwd=fwd, bwd=bwd, total=index + fwd + bwd)


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r.strip().split(",") for r in self.file.read().strip().splitlines() if r.strip()]
        os.unlink(self.file.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def traffic_record(kernel_file: str, workload: str):
    """Per-launch DRAM bytes from a committed ncu summary, if it still matches the source and the workload."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f)
    src = os.path.join(ROOT, "block_sparse_attention_scores_gb300", "csrc", kernel_file)
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    r = rec.get(kernel_file)
    if not r or r.get("source_sha") != sha or r.get("workload") != workload:
        return None
    return r


# ----------------------------------------------------------------------------- multi-rank helpers
def dist_max(value: float, device=None) -> float:
    """Max of a per-rank value over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_workload(w, rank: int):
    """Each rank runs its own batch: same shapes, its own seed (weak scaling)."""
    return w.with_(seed=w.seed + 1000 * rank)


def aggregate_tokens_per_s(w, world: int, max_ms_per_step: float) -> float:
    """Whole-job throughput: tokens of all ranks over the slowest rank's step time."""
    return w.B * w.T * world / (max_ms_per_step * 1e-3)


# ----------------------------------------------------------------------------- CPU oracle baseline
def oracle_sample(w, seconds: float, seed: int = 0):
    """Time the fp64 oracle on a bounded sample of the workload and extrapolate.

    Sample: R query rows (b, g, t) drawn uniformly, run through the oracle's
    index top-k, forward (all heads of the group) and per-query backward; plus
    one of the last four KV blocks through the per-block backward (dK, dV,
    dk_idx), whose cost scales with the number of (row, block) selections. Whole-step oracle time =
    (B*G*T / R) * t_rows + (B*G*T*k / E) * t_block, E = selections of that block.
    Returns (tokens_per_s, description, threads).
    """
    import numpy as np

    import oracle

    rng = np.random.default_rng(seed)
    s = oracle.shape_of(w)
    # inputs: only what the sample touches must be right, but the oracle reads
    # whole tensors, so draw them all (seeded, same generator as the GPU arm)
    inp = synth.make_inputs(w)
    bi = synth.synthetic_block_idx(w)
    hg = w.Hq // w.G
    R = 8
    t0 = time.perf_counter()
    t_rows = 0.0
    rows_done = 0
    while True:
        b = rng.integers(0, w.B, R)
        g = rng.integers(0, w.G, R)
        t = rng.integers(0, w.T, R)
        rows = (b * w.G + g) * w.T + t
        a = time.perf_counter()
        oracle.index_topk(s, inp["q_idx"], inp["k_idx"], rows=rows)
        hrows = ((b * w.T + t)[:, None] * w.Hq + (g * hg)[:, None] + np.arange(hg)[None, :]).ravel()
        oracle.sparse_fwd(s, inp["Q"], inp["K"], inp["V"], bi, rows=hrows)
        oracle.bwd_rows(s, *[inp[n] for n in ("Q", "K", "V", "dO", "q_idx", "k_idx")], bi, rows=rows)
        t_rows += time.perf_counter() - a
        rows_done += R
        if time.perf_counter() - t0 > 0.6 * seconds:
            break
    # one of the last four KV blocks: selected mostly by its own 128 queries per
    # group, which bounds the sample; per selection it costs what any block costs
    c = int(w.n_blocks - 1 - rng.integers(0, min(4, w.n_blocks)))
    b0 = int(rng.integers(0, w.B))
    a = time.perf_counter()
    oracle.bwd_blocks(s, *[inp[n] for n in ("Q", "K", "V", "dO", "q_idx", "k_idx")], bi, blocks=[b0 * w.n_blocks + c])
    t_block = time.perf_counter() - a
    E = int((bi[b0] == c).sum())
    total = (w.B * w.G * w.T / rows_done) * t_rows + (w.B * w.G * w.T * w.k / max(E, 1)) * t_block
    desc = (f"{rows_done} random queries (b,g,t) through index top-k + forward + per-query backward, and KV block "
            f"{c} (selected {E} times) through the per-block backward; whole step extrapolated by row and "
            f"selection counts ({t_rows + t_block:.1f} s measured)")
    return w.B * w.T / total, desc, oracle.num_threads()


def selection_check(w, host, rows, got, tie_eps=1e-4):
    """The step's block_idx on sampled rows (b, g, t) against the oracle's
    selection from the same seeded q_idx, k_idx: bit-exact except rows whose
    oracle k-th / (k+1)-th pooled scores are closer than tie_eps (counted)."""
    import numpy as np

    import oracle

    want, gap, _ = oracle.index_topk(oracle.shape_of(w), host["q_idx"], host["k_idx"], rows=rows)
    diff = np.any(np.asarray(got) != want, axis=1)
    tie = gap < tie_eps
    return {"rows": int(len(rows)), "near_ties": int(tie.sum()), "mismatch_outside_ties": int((diff & ~tie).sum()),
            "mismatch_in_ties": int((diff & tie).sum()), "tie_eps": tie_eps,
            "note": "192 random rows plus the last 64 queries of group 0, batch 0, compared with oracle steps 1-3"}


def oracle_single_thread(w, seconds: float):
    """The same oracle sample as the cpu_baseline, on one host thread."""
    import oracle

    n = oracle.num_threads()
    oracle.set_num_threads(1)
    try:
        v, desc, _ = oracle_sample(w, seconds, seed=1)
    finally:
        oracle.set_num_threads(n)
    return v, desc


def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    vals = []
    desc, cores = "", 0
    seconds = max(2.0, 60.0 / max(1, args.steps + args.warmup))
    for i in range(args.warmup + args.steps):
        v, desc, cores = oracle_sample(w, seconds, seed=i)
        if i >= args.warmup:
            vals.append(v)
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": w.B * w.T / value * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(w, args.gpus),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def config_dict(w, n):
    return {"workload": w.name, "B": w.B, "T": w.T, "Hq": w.Hq, "G": w.G, "d": w.d, "d_idx": w.d_idx, "Bk": w.Bk,
            "k": w.k, "global_batch": w.B * n, "seq_len": w.T, "parallelism": f"batch-sharded x{n}, no collective",
            "l2": "inputs larger than L2 (Q and dO are 1 GiB each at T=131072)"}


# ----------------------------------------------------------------------------- GPU arm
def run_gpu(args, w):
    import numpy as np
    import torch

    import block_sparse_attention_scores_gb300 as msa

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    s = msa.Shape(B=w.B, T=w.T, Hq=w.Hq, G=w.G, d=w.d, d_idx=w.d_idx, Bk=w.Bk, k=w.k)
    # inputs: seeded synthetic data (each rank its own batch), built on the host once
    ww = rank_workload(w, rank)
    host = synth.make_inputs(ww)

    def pinned(x):
        t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16)
        return t.pin_memory()

    h_in = {n: pinned(host[n]) for n in ("Q", "K", "V", "dO", "q_idx", "k_idx")}
    d_in = {n: h_in[n].to(dev, non_blocking=False) for n in h_in}
    ws = msa.alloc_workspace(s, msa.MSA_WS_BWD, dev)
    bi = torch.empty((w.B, w.G, w.T, w.k), dtype=torch.int32, device=dev)
    O = torch.empty_like(d_in["Q"])
    LSE = torch.empty((w.B, w.T, w.Hq), dtype=torch.float32, device=dev)
    f32 = dict(dtype=torch.float32, device=dev)
    out = dict(dQ=torch.empty(d_in["Q"].shape, **f32), dK=torch.empty(d_in["K"].shape, **f32),
               dV=torch.empty(d_in["V"].shape, **f32), dq_idx=torch.empty(d_in["q_idx"].shape, **f32),
               dk_idx=torch.empty(d_in["k_idx"].shape, **f32), KL=torch.empty((w.B, w.G, w.T), **f32))
    stream = torch.cuda.current_stream(dev)
    ev = {}

    timed = (("index_topk", msa.MSA_TIME_INDEX_TOPK), ("sparse_fwd", msa.MSA_TIME_SPARSE_FWD),
             ("bwd", msa.MSA_TIME_BWD))

    def step(d, record=False, kev=None):
        if kev:  # the library records these around each stage's main kernel
            for name, which in timed:
                msa.msa_set_timing_events(which, *kev[name])
        if record:
            ev["a"].record(stream)
        msa.msa_index_topk(s, d["q_idx"], d["k_idx"], bi, ws, stream)
        if record:
            ev["b"].record(stream)
        # one inverted block map of this step's selection serves the forward and the backward
        msa.msa_block_map(s, bi, ws, stream)
        msa.msa_sparse_fwd_mapped(s, d["Q"], d["K"], d["V"], bi, O, LSE, ws, stream)
        if record:
            ev["c"].record(stream)
        msa.msa_bwd_mapped(s, d["Q"], d["K"], d["V"], O, d["dO"], LSE, d["q_idx"], d["k_idx"], bi, 1.0, out["dQ"],
                    out["dK"], out["dV"], out["dq_idx"], out["dk_idx"], out["KL"], ws, stream)
        if record:
            ev["d"].record(stream)

    for _ in range(args.warmup):
        step(d_in)
    msa.msa_check_device_status(ws, stream)
    torch.cuda.synchronize()

    # ---- device-resident timing, per-phase events inside the timed region
    phase = {"index_topk": [], "sparse_fwd": [], "bwd": []}
    clocks = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if clocks:
        clocks.start()
        time.sleep(0.5)
    launches0 = msa.msa_kernel_launches()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    steps_ev = []
    steps_kev = []
    for _ in range(args.steps):
        kev = {name: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for name, _ in timed}
        for pair in kev.values():
            for x in pair:
                x.record(stream)  # creates the event; the library re-records it around the kernel
        steps_kev.append(kev)
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(args.steps):
        ev = {k: torch.cuda.Event(enable_timing=True) for k in "abcd"}
        step(d_in, record=True, kev=steps_kev[i])
        steps_ev.append(ev)
    e1.record(stream)
    torch.cuda.synchronize()
    for _, which in timed:
        msa.msa_set_timing_events(which, None, None)
    if dist:
        dist.barrier()
    launches = msa.msa_kernel_launches() - launches0
    clk = clocks.stop() if clocks else None
    total_ms = e0.elapsed_time(e1)
    for ev in steps_ev:
        phase["index_topk"].append(ev["a"].elapsed_time(ev["b"]))
        phase["sparse_fwd"].append(ev["b"].elapsed_time(ev["c"]))
        phase["bwd"].append(ev["c"].elapsed_time(ev["d"]))
    kernel_ms = {name: statistics.mean(k[name][0].elapsed_time(k[name][1]) for k in steps_kev) for name, _ in timed}
    msa.msa_check_device_status(ws, stream)
    total_ms = dist_max(total_ms, dev)
    ms_step = total_ms / args.steps

    # ---- IndexShare: a layer that reuses an earlier layer's selection and
    # block map (built once, outside the timed region) runs only the mapped
    # forward and backward
    msa.msa_block_map(s, bi, ws, stream)
    for _ in range(2):
        msa.msa_sparse_fwd_mapped(s, d_in["Q"], d_in["K"], d_in["V"], bi, O, LSE, ws, stream)
        msa.msa_bwd_mapped(s, d_in["Q"], d_in["K"], d_in["V"], O, d_in["dO"], LSE, d_in["q_idx"], d_in["k_idx"], bi,
                           1.0, out["dQ"], out["dK"], out["dV"], out["dq_idx"], out["dk_idx"], out["KL"], ws, stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    g0 = torch.cuda.Event(enable_timing=True)
    g1 = torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for _ in range(args.steps):
        msa.msa_sparse_fwd_mapped(s, d_in["Q"], d_in["K"], d_in["V"], bi, O, LSE, ws, stream)
        msa.msa_bwd_mapped(s, d_in["Q"], d_in["K"], d_in["V"], O, d_in["dO"], LSE, d_in["q_idx"], d_in["k_idx"], bi,
                           1.0, out["dQ"], out["dK"], out["dV"], out["dq_idx"], out["dk_idx"], out["KL"], ws, stream)
    g1.record(stream)
    torch.cuda.synchronize()
    share_ms = dist_max(g0.elapsed_time(g1) / args.steps, dev)
    msa.msa_check_device_status(ws, stream)

    # ---- end to end through the C ABI with host buffers (copies inside the timed region).
    # Every step copies all six inputs host->device from pinned memory and
    # reads its result, the per-query KL loss, device->host; the gradients and
    # O stay on the device, where the rest of a training step consumes them.
    # The copies run on their own streams, double-buffered, so step i+1's
    # inputs and step i's result move while step i computes.
    h_kl = [torch.empty(out["KL"].shape, dtype=out["KL"].dtype, pin_memory=True) for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in h_in.values())
    d2h = h_kl[0].numel() * h_kl[0].element_size()
    d_e2e = [{n: torch.empty_like(d_in[n]) for n in d_in} for _ in range(2)]
    o_e2e = [dict(out, O=O)] + [{n: torch.empty_like(t) for n, t in dict(out, O=O).items()}]
    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]    # inputs of buffer b are on the device
    ev_used = [torch.cuda.Event() for _ in range(2)]  # compute on buffer b is done
    ev_out = [torch.cuda.Event() for _ in range(2)]   # outputs of buffer b are on the host

    def step_on(b):
        o = o_e2e[b]
        d = d_e2e[b]
        msa.msa_index_topk(s, d["q_idx"], d["k_idx"], bi, ws, stream)
        msa.msa_block_map(s, bi, ws, stream)
        msa.msa_sparse_fwd_mapped(s, d["Q"], d["K"], d["V"], bi, o["O"], LSE, ws, stream)
        msa.msa_bwd_mapped(s, d["Q"], d["K"], d["V"], o["O"], d["dO"], LSE, d["q_idx"], d["k_idx"], bi, 1.0, o["dQ"],
                    o["dK"], o["dV"], o["dq_idx"], o["dk_idx"], o["KL"], ws, stream)

    def e2e_run(n_steps):
        for i in range(n_steps):
            b = i & 1
            with torch.cuda.stream(s_in):
                s_in.wait_event(ev_used[b])  # step i - 2 has finished reading buffer b
                for n in h_in:
                    d_e2e[b][n].copy_(h_in[n], non_blocking=True)
                ev_in[b].record(s_in)
            stream.wait_event(ev_in[b])
            stream.wait_event(ev_out[b])  # step i - 2's outputs have left buffer b
            step_on(b)
            ev_used[b].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_used[b])
                h_kl[b].copy_(o_e2e[b]["KL"], non_blocking=True)
                ev_out[b].record(s_out)

    e2e_run(2)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    f0 = torch.cuda.Event(enable_timing=True)
    f1 = torch.cuda.Event(enable_timing=True)
    f0.record(s_in)
    stream.wait_event(f0)
    e2e_run(args.steps)
    s_out.wait_stream(stream)
    f1.record(s_out)
    torch.cuda.synchronize()
    e2e_ms = dist_max(f0.elapsed_time(f1) / args.steps, dev)
    msa.msa_check_device_status(ws, stream)
    # the same host->device copies by themselves: this box's pinned-copy rate
    torch.cuda.synchronize()
    c0 = torch.cuda.Event(enable_timing=True)
    c1 = torch.cuda.Event(enable_timing=True)
    c0.record(s_in)
    for i in range(args.steps):
        with torch.cuda.stream(s_in):
            for n in h_in:
                d_e2e[i & 1][n].copy_(h_in[n], non_blocking=True)
    c1.record(s_in)
    torch.cuda.synchronize()
    h2d_ms = c0.elapsed_time(c1) / args.steps
    # rows of this step's selection for the sampled check against the oracle (rank 0, after timing)
    sel_rows = np.random.default_rng(7).integers(0, w.B * w.G * w.T, 192)
    sel_rows = np.concatenate([sel_rows, np.arange(w.T - 64, w.T)])  # the last queries see every block
    sel_got = bi.reshape(-1, w.k)[torch.from_numpy(sel_rows).to(dev)].cpu().numpy()

    # ---- FP8 index top-k (E4M3 copies of q_idx and k_idx, kind::f8f6f4 MMAs) on the same inputs
    ws8 = msa.alloc_workspace(s, msa.MSA_WS_TOPK_FP8, dev)
    bi8 = torch.empty_like(bi)
    for _ in range(2):
        msa.msa_index_topk_fp8(s, d_in["q_idx"], d_in["k_idx"], bi8, ws8, stream)
    torch.cuda.synchronize()
    h0 = torch.cuda.Event(enable_timing=True)
    h1 = torch.cuda.Event(enable_timing=True)
    h0.record(stream)
    for _ in range(args.steps):
        msa.msa_index_topk_fp8(s, d_in["q_idx"], d_in["k_idx"], bi8, ws8, stream)
    h1.record(stream)
    torch.cuda.synchronize()
    fp8_ms = dist_max(h0.elapsed_time(h1) / args.steps, dev)
    msa.msa_check_device_status(ws8, stream)
    del ws8, bi8

    # ---- indexer warmup: full causal attention and the KL against the dense teacher at this workload,
    # through msa_dense_fwd + msa_dense_bwd (outputs in the step's buffers). A step is about a second at
    # T = 131072: at most three timed steps.
    warm = None
    if w.Hq // w.G in (4, 8):
        sd = msa.Shape(B=w.B, T=w.T, Hq=w.Hq, G=w.G, d=w.d, d_idx=w.d_idx, Bk=w.Bk, k=1)
        wsd = msa.alloc_workspace(sd, msa.MSA_WS_DENSE, dev)
        dkev = {n: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for n in ("fwd", "bwd")}
        for pair in dkev.values():
            for x in pair:
                x.record(stream)

        def dense_step():
            msa.msa_dense_fwd(sd, d_in["Q"], d_in["K"], d_in["V"], O, LSE, wsd, stream)
            msa.msa_dense_bwd(sd, d_in["Q"], d_in["K"], d_in["V"], O, d_in["dO"], LSE, d_in["q_idx"], d_in["k_idx"],
                              1.0, out["dQ"], out["dK"], out["dV"], out["dq_idx"], out["dk_idx"], out["KL"], wsd,
                              stream)

        for _ in range(args.warmup):
            dense_step()
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        n_dense = min(args.steps, 3)
        msa.msa_set_timing_events(msa.MSA_TIME_DENSE_FWD, *dkev["fwd"])
        msa.msa_set_timing_events(msa.MSA_TIME_DENSE_BWD, *dkev["bwd"])
        u0 = torch.cuda.Event(enable_timing=True)
        u1 = torch.cuda.Event(enable_timing=True)
        u0.record(stream)
        for _ in range(n_dense):
            dense_step()
        u1.record(stream)
        torch.cuda.synchronize()
        msa.msa_set_timing_events(msa.MSA_TIME_DENSE_FWD, None, None)
        msa.msa_set_timing_events(msa.MSA_TIME_DENSE_BWD, None, None)
        msa.msa_check_device_status(wsd, stream)
        warm_ms = dist_max(u0.elapsed_time(u1) / n_dense, dev)
        wk = {n: dkev[n][0].elapsed_time(dkev[n][1]) for n in dkev}  # the last step's kernels
        del wsd
        ns = w.B * w.G * w.T * (w.T + 1) // 2  # causal (query, key) pairs
        fwd_fl = 4 * w.d * (w.Hq // w.G) * ns
        bwd_fl = 10 * w.d * (w.Hq // w.G) * ns + 6 * w.d_idx * ns
        warm = {"workload": w.name.rsplit("_k", 1)[0] + "_full_attention", "steps": n_dense,
                "ms_per_step": warm_ms, "tokens_per_s": aggregate_tokens_per_s(w, world, warm_ms),
                "tflops": (fwd_fl + bwd_fl) / (warm_ms * 1e-3) / 1e12,
                "dense_fwd_kernel": {"ms": wk["fwd"], "tflops": fwd_fl / (wk["fwd"] * 1e-3) / 1e12},
                "bwd_wide_kernel_dense": {"ms": wk["bwd"], "tflops": bwd_fl / (wk["bwd"] * 1e-3) / 1e12},
                "note": "indexer warmup at this workload: msa_dense_fwd + msa_dense_bwd (every visible token, "
                        "KL against the dense teacher); counted FLOPs as for the sparse step over the T(T+1)/2 "
                        "causal pairs; kernel times from CUDA events of the last timed step"}

    if rank == 0:
        fl = counted_flops(w)
        ab = algorithmic_bytes(w)
        peaks, src = measured_peaks()
        tokens = w.B * w.T * world
        tflops = fl["total"] / (ms_step * 1e-3) / 1e12
        pm = {k: statistics.mean(v) for k, v in phase.items()}
        # Denominators: the burst bf16 figure (a kernel or a step of tens of ms at full SM clock), with the
        # sustained one (seconds of back-to-back GEMMs under the power cap) reported beside it.
        peak = float(peaks.get("bf16_tflops", 1900.0))
        peak_sus = float(peaks.get("bf16_tflops_sustained", peak))
        hbm = float(peaks.get("hbm_gbs", 6800.0))
        # dominant kernel of the step, timed alone (events recorded by the library around its launches)
        stage_flops = {"index_topk": fl["index"], "sparse_fwd": fl["fwd"], "bwd": fl["bwd"]}
        stage_bytes = {"index_topk": ab["index"], "sparse_fwd": ab["fwd"], "bwd": ab["bwd"]}
        wide = w.Hq // w.G >= 4  # 4 or 8 heads per group: the 128-row-tile backward
        kname = {"index_topk": "index_topk_kernel", "sparse_fwd": "sparse_fwd_kernel",
                 "bwd": "bwd_wide_kernel" if wide else "bwd_kernel"}
        kfile = {"index_topk": "index_topk.cu", "sparse_fwd": "sparse_fwd.cu",
                 "bwd": "sparse_bwd_wide.cu" if wide else "sparse_bwd.cu"}
        dom = max(kernel_ms, key=kernel_ms.get)
        achieved = stage_flops[dom] / (kernel_ms[dom] * 1e-3) / 1e12
        kernels_line = {}
        for n in kernel_ms:
            sec = kernel_ms[n] * 1e-3
            tr_n = traffic_record(kfile[n], w.name)
            kernels_line[kname[n]] = {
                "ms": kernel_ms[n], "tflops": stage_flops[n] / sec / 1e12,
                "frac_bf16_peak": stage_flops[n] / sec / 1e12 / peak,
                "algorithmic_gb": stage_bytes[n] / 1e9,
                "algorithmic_gbs": stage_bytes[n] / sec / 1e9,
                "dram_gb_measured": tr_n["bytes_per_launch"] / 1e9 if tr_n else None,
                "dram_gbs_measured": tr_n["bytes_per_launch"] / sec / 1e9 if tr_n else None,
                "frac_hbm_measured": tr_n["bytes_per_launch"] / sec / 1e9 / hbm if tr_n else None}
        tr = traffic_record(kfile[dom], w.name)
        line = {
            "metric": METRIC, "value": aggregate_tokens_per_s(w, world, ms_step), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": config_dict(w, world),
            "step": "msa_index_topk -> msa_block_map -> msa_sparse_fwd_mapped -> msa_bwd_mapped (one block map "
                    "of the step's selection serves both passes)",
            "tflops": tflops, "frac_bf16_peak": tflops / peak, "frac_bf16_peak_sustained": tflops / peak_sus,
            "fwd_tokens_per_s": tokens / ((pm["index_topk"] + pm["sparse_fwd"]) * 1e-3),
            "phases_ms": pm,
            "kernels": kernels_line,
            "counted_flops_per_step": fl["total"] * world,
            "algorithmic_bytes_per_step": ab["total"] * world,
            "roofline": {"kernel": f"{kname[dom]} ({kfile[dom]}), CUDA events around each launch",
                         "bound": "tensor", "achieved": achieved,
                         "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                         "peak_source": (f"{src} bf16 burst (MEASURED_PEAKS.json bf16_tflops)" if src == "measured"
                                         else "fallback 1.9 PFLOP/s bf16 burst"),
                         "peak_sustained": peak_sus, "frac_sustained": achieved / peak_sus,
                         "traffic": tr["bytes_per_launch"] if tr else None,
                         "algorithmic_bytes": stage_bytes[dom],
                         "traffic_over_algorithmic": tr["bytes_per_launch"] / stage_bytes[dom] if tr else None},
            "e2e": {"value": aggregate_tokens_per_s(w, world, e2e_ms), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                    "h2d_gbs_alone": h2d / (h2d_ms * 1e-3) / 1e9, "h2d_ms_alone": h2d_ms,
                    "note": "per step: all inputs host->device (pinned) and the KL loss device->host, on their own "
                            "streams, double-buffered: step i+1's inputs and step i's loss move while step i "
                            "computes; the gradients and O stay on the device. h2d_*_alone: the same copies "
                            "timed by themselves on this box"},
            "clocks": clk,
            "gpu_launches": launches,
            "index_share": {"ms_per_layer": share_ms, "tokens_per_s": aggregate_tokens_per_s(w, world, share_ms),
                            "tflops": (fl["fwd"] + fl["bwd"]) / (share_ms * 1e-3) / 1e12,
                            "note": "a layer reusing an earlier layer's block_idx and block map "
                                    "(msa_block_map once): msa_sparse_fwd_mapped + msa_bwd_mapped"},
            "index_topk_fp8": {"ms": fp8_ms, "tflops": fl["index"] / (fp8_ms * 1e-3) / 1e12,
                               "note": "msa_index_topk_fp8: E4M3 q_idx (per row) and k_idx (per block) with "
                                       "kind::f8f6f4 MMAs; same workload as index_topk"},
            "indexer_warmup": warm,
        }
        if world == 1 and not args.no_cpu_baseline:
            line["selection_check"] = selection_check(w, host, sel_rows, sel_got)
            v, desc, cores = oracle_sample(w, args.cpu_seconds)
            line["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": desc}
            v1, desc1 = oracle_single_thread(w, args.cpu_seconds / 4)
            line["cpu_baseline"]["single_thread"] = {"value": v1, "unit": "tokens/s", "cores": 1, "sample": desc1}
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", type=int, default=3, help="workload preset 0-4 (default 3: T=131072)")
    ap.add_argument("--seq", type=int, default=0, help="override the preset's sequence length (profiling cases)")
    ap.add_argument("--impl", choices=("gb300", "reference"), default="gb300")
    ap.add_argument("--cpu-seconds", type=float, default=20.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    w = synth.CONFIGS[args.config]
    if args.seq:
        w = w.with_(T=args.seq, name=f"{w.name.split('_t')[0]}_t{args.seq}_{w.name.split('_', 3)[-1]}")
    if args.impl == "reference":
        return run_reference(args, w)
    return run_gpu(args, w)


if __name__ == "__main__":
    sys.exit(main())
