"""Benchmark of the paged decode hot path on GB300.

One step = one decode step of the Llama-3-8B-shaped workload (64 sequences,
32 q / 8 kv heads, head_dim 128, bf16, block size 16, context lengths
U[512, 4096], blocks drawn at random from a pool of 1.2x the need): append of
one new token per sequence, then split-K paged decode attention whose
log-sum-exp merge runs inside the same kernel — every kernel of the path,
through the C ABI.

Prints one JSON line (rank 0). `value` is algorithmic KV-cache GB/s of the
whole step (bytes the method must move: every context token's K and V row,
q in and out, table entries, lengths, and the appended rows), measured on the
device with inputs resident in HBM. L2 hygiene: the step cycles through
three copies of the workload (3 x 0.73 GB, > L2), so each step reads its
cache cold. `roofline` reports the split-K kernel alone against the measured
HBM copy bandwidth. `e2e` is the same metric through the same public API with
the step's inputs copied from pinned host memory and the result read back
every step. `cpu_baseline` times the fp64 CPU oracle on a sample of the same
workload.

--impl reference runs the oracle (the only other implementation of this
path) on the host cores as the reference arm.
Multi-GPU (--gpus N under torchrun): independent replicas, one workload per
rank, no collective on the data path (weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from paged_kv_cache_47_gb300 import workloads as W  # noqa: E402

WORKLOAD_INDEX = 1
METRIC = "paged decode attention KV GB/s and seq-tokens/s; fraction of GB300 HBM peak"
UNIT = "GB/s"
KERNEL_SOURCES = ["decode_kernel.cuh", "device_utils.cuh", "decomp.h", "pkv_internal.h"]
PROFILE = os.path.join(ROOT, "profiles", "decode_split_kernel_llama3_8b.md")


# ------------------------------------------------------------------ helpers
def unique_kv_bytes(st, spec):
    """K/V bytes of the distinct physical rows the step reads (a block shared
    by several sequences counted once)."""
    es = torch.tensor([], dtype=W.DTYPES[spec.dtype]).element_size()
    B = spec.block_size
    rows = {}
    for s, L in enumerate(st.context_lens.tolist()):
        for j in range(-(-L // B)):
            b = int(st.block_tables[s, j])
            rows[b] = max(rows.get(b, 0), min(B, L - j * B))
    return sum(rows.values()) * 2 * spec.num_kv_heads * spec.head_dim * es


def step_bytes(st, spec):
    """Algorithmic bytes of one decode step (decode + append)."""
    es = torch.tensor([], dtype=W.DTYPES[spec.dtype]).element_size()
    lens = st.context_lens.long()
    S = lens.numel()
    kv = int(lens.sum()) * 2 * spec.num_kv_heads * spec.head_dim * es
    qo = S * spec.num_q_heads * spec.head_dim * es * 2
    tables = int(((lens + spec.block_size - 1) // spec.block_size).sum()) * 4
    decode = kv + qo + tables + 4 * S
    append = S * spec.num_kv_heads * spec.head_dim * es * 2 * 2 + 8 * S
    return decode, append


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_source_hash():
    """Hash of the decode kernel's code, comments and blank lines left out, so
    that a committed ncu summary stays valid until the code itself changes."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "paged_kv_cache_47_gb300", "csrc", name)) as f:
            text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
        for line in text.splitlines():
            line = line.split("//", 1)[0].rstrip()
            if line:
                h.update(line.encode() + b"\n")
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch of the split-K kernel from the committed ncu
    summary, if it was taken on the current kernel sources."""
    if not os.path.exists(PROFILE):
        return None
    vals = {}
    for line in open(PROFILE):
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            m = re.search(r"`([^`]*)`", v)
            vals[k.strip()] = m.group(1) if m else v.strip()
    if vals.get("kernel_source_hash") != kernel_source_hash():
        return None
    try:
        return float(vals["dram_bytes_per_launch_full_size"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self, t0=None, t1=None):
        """Summarise samples whose timestamp falls in [t0, t1] (host wall
        clock, seconds since the epoch; all samples if not given)."""
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        import datetime
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                f_sm, f_mx = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            if t0 is not None and not (t0 - 0.05 <= ts <= t1 + 0.05):
                continue
            sm.append(f_sm)
            mx = f_mx
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(x: float, world: int, device) -> float:
    """Max of x over all ranks (the slowest rank sets the job's time)."""
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(bytes_per_rank_step: int, steps: int, max_rank_seconds: float, world: int) -> float:
    """Whole-job GB/s: every rank moves bytes_per_rank_step per step (replicas,
    weak scaling) and the job takes as long as its slowest rank."""
    return world * bytes_per_rank_step * steps / max_rank_seconds / 1e9


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ oracle timing
def host_inputs_from_generator(st, seed, device):
    """The step's inputs, re-drawn from the seeded generator and copied to the
    host, with the oracle's own append applied (post-append cache state)."""
    from oracle import oracle

    v = W.make_values(st, seed, device=device)
    h = {k: t.cpu() for k, t in v.items()}
    del v
    oracle.append(h["k_new"], h["v_new"], st.slot_mapping, h["k_pool"], h["v_pool"])
    return h


def time_oracle(st, spec, h, target_s, seq_ids=None):
    """Time oracle decode over the sequences `seq_ids` (all if None), repeated
    until at least target_s of wall time; returns (GB/s, seq-tok/s, s, reps)."""
    from oracle import oracle

    ids = list(range(st.context_lens.numel())) if seq_ids is None else list(seq_ids)
    lens = [int(st.context_lens[i]) for i in ids]
    es = h["q"].element_size()
    nbytes = (sum(lens) * 2 * spec.num_kv_heads * spec.head_dim * es
              + len(ids) * spec.num_q_heads * spec.head_dim * es * 2
              + sum((L + spec.block_size - 1) // spec.block_size for L in lens) * 4 + 4 * len(ids))
    scale = 1.0 / math.sqrt(spec.head_dim)
    spent, reps = 0.0, 0
    while spent < target_s or reps == 0:
        t0 = time.perf_counter()
        oracle.decode(h["q"], h["k_pool"], h["v_pool"], st.block_tables, st.context_lens, scale,
                      seq_ids=ids)
        spent += time.perf_counter() - t0
        reps += 1
    return nbytes * reps / spent / 1e9, sum(lens) * reps / spent, spent, reps


# ------------------------------------------------------------------ reference arm
def run_reference(args):
    world, rank, local = dist_env()
    if rank != 0:
        return 0
    from oracle import build_oracle, oracle
    build_oracle.build()
    spec = W.SPECS[WORKLOAD_INDEX]
    st = W.make_structure(spec, args.seed)
    # bounded sample: the first `ref_seqs` sequences of the workload, values
    # drawn on the host (no GPU involved in this arm)
    n = min(args.ref_seqs, st.context_lens.numel())
    lens = st.context_lens[:n].tolist()
    sub = W.WorkloadSpec("sample", n, spec.num_q_heads, spec.num_kv_heads, spec.head_dim,
                         spec.block_size, spec.dtype, spec.std)
    sst, v = W.make_workload(sub, seed=args.seed, lengths=lens)
    oracle.append(v["k_new"], v["v_new"], sst.slot_mapping, v["k_pool"], v["v_pool"])
    for _ in range(args.warmup):
        time_oracle(sst, sub, v, 0.0)
    rates, toks, secs = [], [], []
    for _ in range(args.steps):
        r, tps, sec, reps = time_oracle(sst, sub, v, 0.0)
        rates.append(r)
        toks.append(tps)
        secs.append(sec / reps)
    value = statistics.median(rates)
    sample = f"{n} of {st.context_lens.numel()} sequences ({sum(lens)} context tokens) per step"
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1000 * statistics.median(secs), 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(spec, st),
        "seq_tokens_per_s": round(statistics.median(toks), 1),
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def workload_config(spec, st):
    return {"workload": spec.name + "_decode_step", "num_seqs": spec.num_seqs,
            "q_heads": spec.num_q_heads, "kv_heads": spec.num_kv_heads,
            "head_dim": spec.head_dim, "block_size": spec.block_size, "kv_dtype": spec.dtype,
            "context_lens": (f"{spec.shared_prefix}-token shared prefix + U[{spec.suffix_lo},{spec.suffix_hi}]"
                             if spec.shared_prefix else f"U[{spec.len_lo},{spec.len_hi}]")
                            + f" seed 0, sum {int(st.context_lens.sum())}",
            "pool_blocks": st.num_blocks,
            "step": ("pkv_block_copy (copy-on-write) + " if st.cow_pairs.numel() else "")
                    + "pkv_append + pkv_decode_attention (split-K with in-kernel merge)"}


# ------------------------------------------------------------------ our arm
def run_ours(args):
    from paged_kv_cache_47_gb300 import binding, build

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    if rank == 0:
        build.build()
    barrier(world)
    binding.lib()

    spec = W.SPECS[args.workload]
    if args.block_size:
        spec = spec.with_block_size(args.block_size)
    if args.dtype:
        from dataclasses import replace
        spec = replace(spec, dtype=args.dtype)
    st = W.make_structure(spec, args.seed)
    scale = 1.0 / math.sqrt(spec.head_dim)
    vals = W.make_values(st, args.seed, device=dev)
    cow = st.cow_pairs if st.cow_pairs.numel() else None
    tables = st.block_tables.to(dev)
    lens = st.context_lens.to(dev)
    slots = st.slot_mapping.to(dev)
    S, Hq, D = vals["q"].shape
    # three resident copies of the cache so every step reads a cold L2
    copies = []
    for c in range(args.copies):
        kp = vals["k_pool"] if c == 0 else vals["k_pool"].clone()
        vp = vals["v_pool"] if c == 0 else vals["v_pool"].clone()
        out = torch.empty(S, Hq, D, dtype=vals["q"].dtype, device=dev)
        ws = binding.alloc_workspace(kp, Hq)
        copies.append((kp, vp, out, ws))
    decode_bytes, append_bytes = step_bytes(st, spec)
    total_bytes = decode_bytes + append_bytes
    if cow is not None:
        es = vals["q"].element_size()
        total_bytes += cow.shape[0] * 2 * 2 * spec.num_kv_heads * spec.block_size * spec.head_dim * es
    # bytes the split-K kernel must bring from HBM: shared blocks once
    hbm_decode_bytes = decode_bytes - (int(st.context_lens.sum()) * 2 * spec.num_kv_heads *
                                       spec.head_dim * vals["q"].element_size()) + \
        unique_kv_bytes(st, spec)
    stream = torch.cuda.current_stream()
    # prepared calls: the C-ABI arguments are marshalled once per cache copy
    calls = []
    for kp, vp, out, ws in copies:
        calls.append((binding.PreparedAppend(vals["k_new"], vals["v_new"], slots, kp, vp),
                      binding.PreparedDecode(vals["q"], kp, vp, tables, lens, scale, out, ws,
                                             consumer=args.consumer)))

    def step(i, evs=None, s=None, aevs=None):
        app, dec = calls[i % len(calls)]
        s = s if s is not None else torch.cuda.current_stream()
        if aevs is not None:
            aevs[0].record(s)
        if cow is not None:      # copy-on-write of the last shared block, then append
            kp, vp = copies[i % len(copies)][:2]
            binding.block_copy(cow, kp, vp, stream=s)
        if aevs is not None:
            aevs[1].record(s)
        app(s)
        if aevs is not None:
            aevs[2].record(s)
        dec(s, timing_events=evs)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if binding.get_error() != 0:
        raise RuntimeError("device error word set during warm-up")

    # per-kernel events on a strided subset of the timed steps
    stride = max(1, args.steps // 200)
    kev = {}
    for i in range(0, args.steps, stride):
        pair = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        for e in pair:
            e.record(stream)            # materialise the CUDA event handle
        kev[i] = pair
    # append and copy-on-write events on the same steps (eager launches only:
    # torch's events are not recorded as nodes of a captured graph)
    aev = {}
    if args.launch == "eager":
        for i in kev:
            trio = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            for e in trio:
                e.record(stream)
            aev[i] = trio
    torch.cuda.synchronize()

    if args.launch == "graph":
        # each step replays a captured graph of the same kernel launches
        def capture(i, evs):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, capture_error_mode="thread_local"):
                step(i, evs)
            return g
        plain = [capture(c, None) for c in range(len(calls))]
        timed = {i: capture(i, kev[i]) for i in kev}
        torch.cuda.synchronize()
        for i in range(3):
            plain[i % len(plain)].replay()
        torch.cuda.synchronize()

        def run_step(i):
            (timed[i] if i in timed else plain[i % len(plain)]).replay()
    else:
        def run_step(i):
            step(i, kev.get(i), aevs=aev.get(i))

    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.15)

    barrier(world)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    epoch0 = time.time()
    t_start.record(stream)
    for i in range(args.steps):
        run_step(i)
    t_end.record(stream)
    enqueue_s = time.perf_counter() - wall0
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    barrier(world)
    clocks = sampler.stop(epoch0, epoch0 + wall)

    ms = t_start.elapsed_time(t_end)
    ms_max = reduce_max(ms, world, dev)
    split_ms = [kev[i][0].elapsed_time(kev[i][1]) for i in kev]
    split_avg = sum(split_ms) / len(split_ms)
    side = {}
    if aev:
        es = vals["q"].element_size()
        app_ms = sum(aev[i][1].elapsed_time(aev[i][2]) for i in aev) / len(aev)
        side["append"] = {"avg_us": round(app_ms * 1000, 3), "bytes": append_bytes,
                          "gbs": round(append_bytes / (app_ms / 1000) / 1e9, 2),
                          "note": "K/V rows read + written, slots read; launched alone"}
        if cow is not None:
            cp_ms = sum(aev[i][0].elapsed_time(aev[i][1]) for i in aev) / len(aev)
            cp_bytes = cow.shape[0] * 2 * 2 * spec.num_kv_heads * spec.block_size * spec.head_dim * es
            side["block_copy"] = {"avg_us": round(cp_ms * 1000, 3), "bytes": cp_bytes,
                                  "gbs": round(cp_bytes / (cp_ms / 1000) / 1e9, 2),
                                  "note": "whole K and V blocks read + written"}
    if binding.get_error() != 0:
        raise RuntimeError("device error word set during the timed region")

    per_step_s = ms_max / 1000.0 / args.steps
    value = job_gbs(total_bytes, args.steps, ms_max / 1000.0, world)
    seq_tok = world * int(st.context_lens.sum()) / per_step_s
    peak, peak_kind = peaks()

    # ------------- end to end: host inputs in, result out, every step
    e2e = run_e2e(args, st, spec, vals, copies, tables, lens, slots, scale, stream, dev,
                  total_bytes, world)

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max / args.steps, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": spec.dtype,
        "data": "synthetic (seeded N(0,1) values, random block tables)",
        "config": {**workload_config(spec, st),
                   "l2": f"inputs > L2: the step cycles through {len(copies)} resident copies "
                         f"of the cache ({len(copies)} x {2 * st.num_blocks * spec.num_kv_heads * spec.block_size * spec.head_dim * 2 / 1e9:.2f} GB)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "launch": "CUDA-graph replay of the step's kernel launches (captured through the C ABI)"
                             if args.launch == "graph" else "eager C-ABI calls"},
        "seq_tokens_per_s": round(seq_tok, 1),
        "hbm_frac_of_measured": round(value / peak / world, 4),
        "roofline": {"bound": "hbm", "kernel": "decode_split_kernel",
                     "achieved": round(hbm_decode_bytes / (split_avg / 1000.0) / 1e9, 2),
                     "peak": peak, "unit": "GB/s",
                     "frac": round(hbm_decode_bytes / (split_avg / 1000.0) / 1e9 / peak, 4),
                     "traffic": profiled_traffic() if args.workload == WORKLOAD_INDEX and not args.block_size else None,
                     "algorithmic_bytes_per_launch": hbm_decode_bytes,
                     "logical_bytes_per_launch": decode_bytes,
                     "avg_launch_ms": round(split_avg, 5),
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"},
        "other_kernels": side or None,
        "gpu_launches": (2 + (1 if cow is not None else 0)) * args.steps,
        "clocks": clocks,
        "wall_s_timed_region": round(wall, 4),
        "host_enqueue_s": round(enqueue_s, 4),
        "e2e": e2e,
    }
    if rank == 0 and not args.no_cpu_baseline:
        from oracle import oracle
        h = host_inputs_from_generator(st, args.seed, dev)
        r, tps, sec, reps = time_oracle(st, spec, h, args.cpu_seconds)
        cores = oracle.num_threads()
        line["cpu_baseline"] = {"value": round(r, 4), "unit": UNIT, "cores": cores,
                                "kind": "oracle", "seq_tokens_per_s": round(tps, 1),
                                "sample": f"the whole workload ({S} sequences, "
                                          f"{int(st.context_lens.sum())} context tokens) x {reps} "
                                          f"repetitions, {sec:.1f} s of fp64 oracle decode"}
        # the same oracle on one core, over the first sequences only
        n1 = min(4, S)
        oracle.set_num_threads(1)
        try:
            r1, tps1, sec1, reps1 = time_oracle(st, spec, h, args.cpu_seconds / 4,
                                                seq_ids=range(n1))
        finally:
            oracle.set_num_threads(cores)
        line["cpu_baseline"]["one_core"] = {
            "value": round(r1, 4), "unit": UNIT, "seq_tokens_per_s": round(tps1, 1),
            "sample": f"first {n1} sequences x {reps1} repetitions, {sec1:.1f} s"}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_e2e(args, st, spec, vals, copies, tables, lens, slots, scale, stream, dev, total_bytes,
            world):
    from paged_kv_cache_47_gb300 import binding

    pin = lambda t: t.detach().cpu().pin_memory()  # noqa: E731
    h_q, h_kn, h_vn = pin(vals["q"]), pin(vals["k_new"]), pin(vals["v_new"])
    h_tab, h_len, h_slot = pin(st.block_tables), pin(st.context_lens), pin(st.slot_mapping)
    d_q, d_kn, d_vn = torch.empty_like(vals["q"]), torch.empty_like(vals["k_new"]), torch.empty_like(vals["v_new"])
    d_tab, d_len, d_slot = torch.empty_like(tables), torch.empty_like(lens), torch.empty_like(slots)
    h_out = torch.empty(vals["q"].shape, dtype=vals["q"].dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (h_q, h_kn, h_vn, h_tab, h_len, h_slot))
    d2h = h_out.numel() * h_out.element_size()
    steps = min(args.steps, args.e2e_steps)

    calls = []
    for kp, vp, out, ws in copies:
        calls.append((binding.PreparedAppend(d_kn, d_vn, d_slot, kp, vp),
                      binding.PreparedDecode(d_q, kp, vp, d_tab, d_len, scale, out, ws), out))

    cow = st.cow_pairs if st.cow_pairs.numel() else None

    def one(i):
        app, dec, out = calls[i % len(calls)]
        for d, h in ((d_q, h_q), (d_kn, h_kn), (d_vn, h_vn), (d_tab, h_tab), (d_len, h_len),
                     (d_slot, h_slot)):
            d.copy_(h, non_blocking=True)
        if cow is not None:
            kp, vp = copies[i % len(copies)][:2]
            binding.block_copy(cow, kp, vp, stream=stream)
        app(stream)
        dec(stream)
        h_out.copy_(out, non_blocking=True)
        stream.synchronize()            # the step's result is on the host

    for i in range(3):
        one(i)
    barrier(world)
    t0 = time.perf_counter()
    for i in range(steps):
        one(i)
    dt = time.perf_counter() - t0
    dt = reduce_max(dt, world, dev)
    return {"value": round(world * total_bytes * steps / dt / 1e9, 2), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "ms_per_step": round(1000 * dt / steps, 4)}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--copies", type=int, default=3)
    ap.add_argument("--e2e-steps", type=int, default=500)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-seqs", type=int, default=16)
    ap.add_argument("--launch", choices=["graph", "eager"], default="eager")
    ap.add_argument("--workload", type=int, default=WORKLOAD_INDEX,
                    help="index of the workload (0 tiny, 1 Llama-3-8B-shaped [default], "
                         "2 OPT-13B-shaped MHA, 3 agent swarm with prefix sharing, "
                         "4 long-context 70B-shaped)")
    ap.add_argument("--block-size", type=int, default=0, help="override the workload's block size")
    ap.add_argument("--dtype", choices=["f32", "f16", "bf16"], default=None,
                    help="override the workload's K/V dtype")
    ap.add_argument("--consumer", type=int, default=0,
                    help="math path: 0 auto, 1 CUDA cores, 2 tensor cores (16-bit only)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
