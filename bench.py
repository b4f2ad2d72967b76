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
import ctypes
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
NOMINAL_HBM_GBS = 8000.0   # GB300 HBM3e, nominal
QUEUE_FILL_CYCLES = 1_000_000   # device sleep (~0.5 ms) before a timed loop's start event
KERNEL_SOURCES = ["decode_kernel.cuh", "device_utils.cuh", "decomp.h", "pkv_internal.h"]
PROFILE = os.path.join(ROOT, "profiles", "decode_split_kernel_llama3_8b.md")


# ------------------------------------------------------------------ helpers
def cache_row_bytes(spec, kv_quant):
    """Bytes of one (token, kv head) row of K (or V) in the cache: D elements,
    or D 8-bit codes plus a 4-byte scale."""
    if kv_quant:
        return spec.head_dim + 4
    return spec.head_dim * torch.tensor([], dtype=W.DTYPES[spec.dtype]).element_size()


def unique_kv_bytes(st, spec, row_bytes):
    """K/V bytes of the distinct physical rows the step reads (a block shared
    by several sequences counted once)."""
    B = spec.block_size
    rows = {}
    for s, L in enumerate(st.context_lens.tolist()):
        for j in range(-(-L // B)):
            b = int(st.block_tables[s, j])
            rows[b] = max(rows.get(b, 0), min(B, L - j * B))
    return sum(rows.values()) * 2 * spec.num_kv_heads * row_bytes


def step_bytes(st, spec, row_bytes, fused=False):
    """Algorithmic bytes of one decode step (decode + append): every context
    row of K and V in the cache, q in and out, table entries, lengths; the
    append reads the new K/V activations and writes their cache rows. With the
    append fused into the decode (fused=True) the decode reads each new row
    from the activations once, for the attention and the write alike, so the
    append part is only the rows written."""
    es = torch.tensor([], dtype=W.DTYPES[spec.dtype]).element_size()
    lens = st.context_lens.long()
    S = lens.numel()
    kv = int(lens.sum()) * 2 * spec.num_kv_heads * row_bytes
    qo = S * spec.num_q_heads * spec.head_dim * es * 2
    tables = int(((lens + spec.block_size - 1) // spec.block_size).sum()) * 4
    decode = kv + qo + tables + 4 * S
    if fused:
        return decode, S * spec.num_kv_heads * 2 * row_bytes
    append = S * spec.num_kv_heads * 2 * (spec.head_dim * es + row_bytes) + 8 * S
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
def host_inputs_from_generator(st, seed, device, kv_quant=None):
    """The step's inputs, re-drawn from the seeded generator and copied to the
    host, with the oracle's own append applied (post-append cache state). For
    an 8-bit cache the oracle quantizes every context row itself."""
    from oracle import oracle

    v = W.make_values(st, seed, device=device)
    h = {k: t.cpu() for k, t in v.items()}
    del v
    oracle.append(h["k_new"], h["v_new"], st.slot_mapping, h["k_pool"], h["v_pool"])
    if kv_quant:
        NB, Hk, B, D = h["k_pool"].shape
        slots = set()
        for s, L in enumerate(st.context_lens.tolist()):
            row = st.block_tables[s].tolist()
            slots.update(row[t // B] * B + t % B for t in range(L))
        sl = torch.tensor(sorted(slots), dtype=torch.int64)
        kr = h["k_pool"][sl // B, :, sl % B].contiguous()
        vr = h["v_pool"][sl // B, :, sl % B].contiguous()
        kc = torch.zeros(NB, Hk, B, D, dtype=torch.uint8)
        ks = torch.zeros(NB, Hk, B, dtype=torch.float32)
        q = {"k_codes": kc, "v_codes": kc.clone(), "k_scales": ks, "v_scales": ks.clone()}
        oracle.append_quant(kv_quant, kr, vr, sl, q["k_codes"], q["v_codes"], q["k_scales"],
                            q["v_scales"])
        h = {"q": h["q"], "quant": kv_quant, **q}
    return h


def time_oracle(st, spec, h, target_s, seq_ids=None):
    """Time oracle decode over the sequences `seq_ids` (all if None), repeated
    until at least target_s of wall time; returns (GB/s, seq-tok/s, s, reps)."""
    from oracle import oracle

    ids = list(range(st.context_lens.numel())) if seq_ids is None else list(seq_ids)
    lens = [int(st.context_lens[i]) for i in ids]
    es = h["q"].element_size()
    row_bytes = cache_row_bytes(spec, h.get("quant"))
    nbytes = (sum(lens) * 2 * spec.num_kv_heads * row_bytes
              + len(ids) * spec.num_q_heads * spec.head_dim * es * 2
              + sum((L + spec.block_size - 1) // spec.block_size for L in lens) * 4 + 4 * len(ids))
    scale = 1.0 / math.sqrt(spec.head_dim)
    spent, reps = 0.0, 0
    while spent < target_s or reps == 0:
        t0 = time.perf_counter()
        if h.get("quant"):
            oracle.decode_quant(h["quant"], h["q"], h["k_codes"], h["v_codes"], h["k_scales"],
                                h["v_scales"], st.block_tables, st.context_lens, scale,
                                seq_ids=ids)
        else:
            oracle.decode(h["q"], h["k_pool"], h["v_pool"], st.block_tables, st.context_lens,
                          scale, seq_ids=ids)
        spent += time.perf_counter() - t0
        reps += 1
    return nbytes * reps / spent / 1e9, sum(lens) * reps / spent, spent, reps


# ------------------------------------------------------------------ block manager
def time_block_manager(st, spec, steps=200):
    """Host cost of the block manager's part of a decode step for this
    workload: one new token for every sequence (pkv_bm_append) and the
    decode tables of the whole batch (pkv_bm_block_tables)."""
    from paged_kv_cache_47_gb300 import binding

    S = st.context_lens.numel()
    B = spec.block_size
    # room for two timed loops of `steps` tokens per sequence
    need = sum(-(-(int(L) + 2 * steps) // B) for L in st.context_lens.tolist())
    bm = binding.BlockManager(need + 8, B)
    for s, L in enumerate(st.context_lens.tolist()):
        bm.add_sequence(s)
        bm.append(s, int(L) - 1)
    M = -(-(int(st.context_lens.max()) + 2 * steps) // B)
    ids = list(range(S))
    ones = [1] * S
    t_app = t_tab = 0.0
    for _ in range(steps):
        t0 = time.perf_counter()
        bm.append_batch(ids, ones)
        t1 = time.perf_counter()
        bm.block_tables(ids, M)
        t_tab += time.perf_counter() - t1
        t_app += t1 - t0
    # the same two calls with their buffers made once: what is left is native
    prep = bm.prepared_step(ids, ones, M)
    p_app = p_tab = 0.0
    for _ in range(steps):
        t0 = time.perf_counter()
        prep.append()
        t1 = time.perf_counter()
        prep.block_tables()
        p_tab += time.perf_counter() - t1
        p_app += t1 - t0
    return {"sequences": S, "append_us_per_step": round(1e6 * t_app / steps, 2),
            "tables_us_per_step": round(1e6 * t_tab / steps, 2),
            "prepared_append_us_per_step": round(1e6 * p_app / steps, 2),
            "prepared_tables_us_per_step": round(1e6 * p_tab / steps, 2),
            "note": "host: one pkv_bm_append_batch and one pkv_bm_block_tables call per "
                    "step, through the Python binding's list-taking calls, then prepared "
                    "(buffers made once, only the two native calls per step)"}


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


def workload_config(spec, st, pending=None, inputs_ready=True, fused=True):
    """The workload and the launch options of its step. pending: whether the
    decode takes pending_tail 1 (default: the 16-bit paged step, which uses it
    unless the step copies blocks); inputs_ready: whether the append reads its
    inputs before its wait; fused: the append runs inside the decode."""
    if pending is None:
        pending = not st.cow_pairs.numel()
    if fused:
        step = (("pkv_block_copy (copy-on-write) + " if st.cow_pairs.numel() else "")
                + "pkv_append_decode_attention (one launch: each sequence's new row taken "
                "from the activations for the attention and written to its slot; split-K "
                "with in-kernel merge; tables_ready: tables and lengths read while the "
                "previous kernel finishes"
                + ("; pending_tail 1: every pool row gathered at once, only the stores wait "
                   "for the previous kernel" if pending else "") + ")")
    else:
        step = None
    return {"workload": spec.name + "_decode_step", "num_seqs": spec.num_seqs,
            "q_heads": spec.num_q_heads, "kv_heads": spec.num_kv_heads,
            "head_dim": spec.head_dim, "block_size": spec.block_size, "kv_dtype": spec.dtype,
            "context_lens": (f"{spec.shared_prefix}-token shared prefix + U[{spec.suffix_lo},{spec.suffix_hi}]"
                             if spec.shared_prefix else f"U[{spec.len_lo},{spec.len_hi}]")
                            + f" seed 0, sum {int(st.context_lens.sum())}",
            "pool_blocks": st.num_blocks,
            "step": step or ("pkv_block_copy (copy-on-write) + " if st.cow_pairs.numel() else "")
                    + "pkv_append"
                    + (" (inputs_ready: it reads its inputs before waiting on the previous "
                       "decode)" if inputs_ready else "")
                    + " + pkv_decode_attention (split-K with in-kernel merge; "
                    "tables_ready: the decode reads tables and lengths while the append "
                    "finishes"
                    + ("; pending_tail 1: it also gathers every row but each sequence's "
                       "appended one meanwhile" if pending else "") + ")"}


# ------------------------------------------------------------------ cache copies
class Pools16:
    """One resident copy of a 16-bit paged cache (K and V pools). fused: the
    step appends inside the decode (pkv_append_decode_attention, one launch)
    instead of a separate pkv_append before it."""

    def __init__(self, kp, vp, fused=True):
        self.kp, self.vp = kp, vp
        self.fused = fused

    def workspace(self, Hq):
        from paged_kv_cache_47_gb300 import binding
        return binding.alloc_workspace(self.kp, Hq)

    def prepared(self, q, kn, vn, slots, tables, lens, scale, out, ws, consumer=0,
                 pending_tail=0):
        from paged_kv_cache_47_gb300 import binding
        if self.fused:
            # one launch: the new rows come from kn / vn (step inputs no kernel
            # writes, read early like q); the tables and lengths are in place
            # before the step (tables_ready)
            return (None, binding.PreparedAppendDecode(q, kn, vn, self.kp, self.vp, tables, lens,
                                                       scale, out, ws, tables_ready=True,
                                                       pending_tail=pending_tail,
                                                       consumer=consumer))
        # the step's tables and lengths are in place before its append runs, so
        # the decode may read them while the append finishes (tables_ready)
        # the new rows and slots are step inputs no kernel writes: the append
        # reads them before it waits for the previous step's decode
        return (binding.PreparedAppend(kn, vn, slots, self.kp, self.vp, inputs_ready=True),
                binding.PreparedDecode(q, self.kp, self.vp, tables, lens, scale, out, ws,
                                       tables_ready=True, pending_tail=pending_tail,
                                       consumer=consumer))

    def cow(self, pairs, stream):
        from paged_kv_cache_47_gb300 import binding
        binding.block_copy(pairs, self.kp, self.vp, stream=stream)

    def clone(self):
        return Pools16(self.kp.clone(), self.vp.clone(), self.fused)


class PoolsQ:
    """One resident copy of an 8-bit paged cache (codes and row scales)."""

    def __init__(self, cache):
        self.cache = cache

    @classmethod
    def fill(cls, code, st, vals, dev):
        """An 8-bit cache holding every context row before the step's append,
        quantized by the library from the drawn activations."""
        from paged_kv_cache_47_gb300 import binding
        NB, Hk, B, D = vals["k_pool"].shape
        cache = binding.QuantCache.empty(NB, Hk, B, D, code, vals["q"].dtype, device=dev)
        slots = set()
        for s, L in enumerate(st.context_lens.tolist()):
            row = st.block_tables[s].tolist()
            slots.update(row[t // B] * B + t % B for t in range(L - 1))
        sl = torch.tensor(sorted(slots), dtype=torch.int64, device=dev)
        blk, off = sl // B, sl % B
        kr = vals["k_pool"][blk, :, off].contiguous()
        vr = vals["v_pool"][blk, :, off].contiguous()
        binding.append_quant(kr, vr, sl, cache)
        torch.cuda.synchronize()
        return cls(cache)

    def workspace(self, Hq):
        from paged_kv_cache_47_gb300 import binding
        return binding.alloc_quant_workspace(self.cache, Hq)

    def prepared(self, q, kn, vn, slots, tables, lens, scale, out, ws, consumer=0,
                 pending_tail=0):
        from paged_kv_cache_47_gb300 import binding
        # pending_tail is not used here: on the 8-bit path, overlapping the
        # next call's start measured 1.7 % slower (mma.sync) and the tensor-core
        # E4M3 step 69.3 -> 69.9 us; int8 88.7 us either way
        return (binding.PreparedAppendQuant(kn, vn, slots, self.cache, inputs_ready=True),
                binding.PreparedDecodeQuant(q, self.cache, tables, lens, scale, out, ws,
                                            tables_ready=True))

    def cow(self, pairs, stream):
        from paged_kv_cache_47_gb300 import binding
        binding.block_copy_quant(pairs, self.cache, stream=stream)

    def clone(self):
        from paged_kv_cache_47_gb300 import binding
        c = self.cache
        return PoolsQ(binding.QuantCache(c.k_codes.clone(), c.v_codes.clone(), c.k_scales.clone(),
                                         c.v_scales.clone(), c.code, c.act_dtype))


class PoolsFlat:
    """One resident copy of a flat cache: one virtual span per sequence, its
    physical chunks mapped as it grows (pkv_flat_*)."""

    def __init__(self, fc, st):
        self.fc, self.st = fc, st

    @classmethod
    def fill(cls, st, vals, dev):
        """Every context row before the step's append, copied into the flat
        spans (slot s = sequence s) by the library's flat append."""
        from paged_kv_cache_47_gb300 import binding
        NB, Hk, B, D = vals["k_pool"].shape
        lens = st.context_lens.tolist()
        cap = -(-max(lens) // 64) * 64
        fc = binding.FlatCache(len(lens), cap, Hk, D, vals["q"].dtype)
        slots, pos, src = [], [], []
        for s, L in enumerate(lens):
            fc.reserve(s, L)
            row = st.block_tables[s].tolist()
            for t in range(L - 1):
                slots.append(s)
                pos.append(t)
                src.append(row[t // B] * B + t % B)
        sl = torch.tensor(src, dtype=torch.int64, device=dev)
        kr = vals["k_pool"][sl // B, :, sl % B].contiguous()
        vr = vals["v_pool"][sl // B, :, sl % B].contiguous()
        fc.append(kr, vr, torch.tensor(slots, dtype=torch.int32, device=dev),
                  torch.tensor(pos, dtype=torch.int32, device=dev))
        torch.cuda.synchronize()
        return cls(fc, st)

    def workspace(self, Hq):
        return self.fc.workspace(Hq)

    def prepared(self, q, kn, vn, slots, tables, lens, scale, out, ws, consumer=0,
                 pending_tail=0):
        S = q.shape[0]
        seq = torch.arange(S, dtype=torch.int32, device=q.device)
        # the appended token sits at position L - 1 (the workload's lengths are fixed)
        pos = (self.st.context_lens - 1).to(torch.int32).to(q.device)
        fc = self.fc

        def app(stream):
            fc.append(kn, vn, seq, pos, stream=stream)

        def dec(stream, timing_events=None):
            fc.decode_attention(q, seq, lens, scale, out=out, workspace=ws,
                                timing_events=timing_events, stream=stream, tables_ready=True,
                                pending_tail=pending_tail)
        return app, dec

    def cow(self, pairs, stream):
        raise RuntimeError("flat spans share no blocks: no copy-on-write")

    def clone(self):
        raise RuntimeError("clone a flat cache by filling a new one")


class PoolsPrefix(Pools16):
    """A 16-bit paged cache decoded prefix-aware: all sequences form one group
    sharing the prefix blocks they still hold in common (one launch of
    pkv_decode_attention_prefix after the separate append)."""

    def __init__(self, kp, vp, shared_blocks):
        super().__init__(kp, vp, fused=False)
        self.shared_blocks = shared_blocks

    def clone(self):
        return PoolsPrefix(self.kp.clone(), self.vp.clone(), self.shared_blocks)

    def workspace(self, Hq):
        return None        # sized per call shape in prepared()

    def prepared(self, q, kn, vn, slots, tables, lens, scale, out, ws, consumer=0,
                 pending_tail=0):
        from paged_kv_cache_47_gb300 import binding
        S = q.shape[0]
        app = binding.PreparedAppend(kn, vn, slots, self.kp, self.vp, inputs_ready=True)
        dec = binding.PreparedDecodePrefix(q, self.kp, self.vp, tables, lens, scale, [0] * S,
                                           [self.shared_blocks], out=out, tables_ready=True,
                                           consumer=consumer)
        return app, dec


# ------------------------------------------------------------------ other workloads
# (workload, block size override, largest suffix override, cache / decode):
# None the 16-bit paged cache and its plain decode, "prefix" the prefix-aware
# decode, "fp8_e4m3" / "int8" the 8-bit cache, "flat" flat spans
SWEEP = [(0, None, None, None), (2, None, None, None), (3, None, None, None),
         (3, None, None, "prefix"), (3, None, 500, None), (3, None, 500, "prefix"),
         (4, 8, None, None), (4, 16, None, None), (4, 32, None, None),
         (1, None, None, "fp8_e4m3"), (1, None, None, "int8"), (1, None, None, "flat"),
         (4, 16, None, "fp8_e4m3"), (4, 16, None, "int8")]
TOL = {"f32": 1e-5, "f16": 2e-3, "bf16": 2e-3}
QUANT = ("fp8_e4m3", "int8")


def workload_sweep(args, dev, peak):
    """Every other workload once, on one resident cache copy (each is larger
    than L2 but the tiny one, which is launch-bound): the step period over
    `steps` back-to-back steps, the decode kernel alone (CUDA events around
    each launch), algorithmic and unique bytes, the fraction of the measured
    peak, and the max-abs error of the whole output against the fp64 oracle
    (every sequence, every head). The Llama-shaped step also runs over the
    8-bit caches and over flat spans, the long-context one over the 8-bit caches."""
    from oracle import oracle
    from paged_kv_cache_47_gb300 import binding

    from dataclasses import replace
    steps = max(args.steps, 10)
    res = []
    for idx, B, suffix_hi, mode in SWEEP:
        prefix_aware, quant = mode == "prefix", mode if mode in QUANT else None
        spec = W.SPECS[idx] if B is None else W.SPECS[idx].with_block_size(B)
        if suffix_hi is not None:
            spec = replace(spec, suffix_hi=suffix_hi)
        st = W.make_structure(spec, args.seed)
        vals = W.make_values(st, args.seed, device=dev)
        h = {k: v.cpu() for k, v in vals.items()}      # the pre-step state, for the oracle
        cow = st.cow_pairs if st.cow_pairs.numel() else None
        tables, lens = st.block_tables.to(dev), st.context_lens.to(dev)
        slots = st.slot_mapping.to(dev)
        S, Hq, D = vals["q"].shape
        scale = 1.0 / math.sqrt(spec.head_dim)
        if prefix_aware:
            # after the copy-on-write the last prefix block is private to all
            # but one holder: the group shares the blocks before it
            pools = PoolsPrefix(vals["k_pool"], vals["v_pool"],
                                spec.shared_prefix // spec.block_size - (1 if cow is not None else 0))
        elif quant:
            pools = PoolsQ.fill(quant, st, vals, dev)
        elif mode == "flat":
            pools = PoolsFlat.fill(st, vals, dev)
        else:
            pools = Pools16(vals["k_pool"], vals["v_pool"])
        fused = isinstance(pools, Pools16) and pools.fused and not prefix_aware
        out = torch.empty(S, Hq, D, dtype=vals["q"].dtype, device=dev)
        ws = pools.workspace(Hq)
        # one cache copy: each step's append rewrites the same last row, so the
        # rows below it are never in flight (pending_tail 1) unless the step
        # copies whole blocks
        app, dec = pools.prepared(vals["q"], vals["k_new"], vals["v_new"], slots, tables, lens,
                                  scale, out, ws, pending_tail=0 if cow is not None else 1)
        stream = torch.cuda.current_stream()

        def step(evs=None):
            if cow is not None:
                pools.cow(cow, stream)
            if app is not None:
                app(stream)
            dec(stream, timing_events=evs)

        for _ in range(3):
            step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(QUEUE_FILL_CYCLES)    # work queued when the start event fires
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        step_ms = e0.elapsed_time(e1) / steps
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
        for pair in evs:
            for e in pair:
                e.record(stream)        # materialise the handles the library records
        torch.cuda.synchronize()
        for pair in evs:
            step(pair)
        torch.cuda.synchronize()
        if binding.get_error() != 0:
            raise RuntimeError(f"device error word set on workload {spec.name}")
        dec_ms = sum(a.elapsed_time(b) for a, b in evs) / steps
        row_bytes = cache_row_bytes(spec, quant)
        decode_bytes, append_bytes = step_bytes(st, spec, row_bytes, fused=fused)
        total = decode_bytes + append_bytes
        if cow is not None:
            total += cow.shape[0] * 2 * 2 * spec.num_kv_heads * spec.block_size * row_bytes
        uniq = decode_bytes - (int(st.context_lens.sum()) * 2 * spec.num_kv_heads * row_bytes) \
            + unique_kv_bytes(st, spec, row_bytes)
        # the oracle on the same inputs: copy-on-write, append, decode of all sequences
        t0 = time.perf_counter()
        if quant:
            # the oracle quantizes every context row (the appended one
            # included) itself, then decodes over its own codes and scales
            hq = host_inputs_from_generator(st, args.seed, dev, quant)
            ref = oracle.decode_quant(quant, hq["q"], hq["k_codes"], hq["v_codes"],
                                      hq["k_scales"], hq["v_scales"], st.block_tables,
                                      st.context_lens, scale)
            del hq
        else:
            if cow is not None:
                oracle.block_copy(cow, h["k_pool"], h["v_pool"])
            oracle.append(h["k_new"], h["v_new"], st.slot_mapping, h["k_pool"], h["v_pool"])
            ref = oracle.decode(h["q"], h["k_pool"], h["v_pool"], st.block_tables,
                                st.context_lens, scale)
        oracle_s = time.perf_counter() - t0
        got = out.double().cpu().numpy()
        err = float(abs(got - ref).max()) if got.size else 0.0
        res.append({
            "workload": spec.name + (f" (suffix U[{spec.suffix_lo},{spec.suffix_hi}])"
                                     if suffix_hi is not None else ""),
            "decode": "prefix-aware (pkv_decode_attention_prefix)" if prefix_aware else
                      (f"8-bit cache: pkv_append_quant_ex + pkv_decode_attention_quant"
                       + (" (tcgen05 kind::f8f6f4)" if quant == "fp8_e4m3" else " (mma.sync)")
                       if quant else
                       "flat spans: pkv_flat_append + pkv_decode_attention_flat"
                       if mode == "flat" else
                       "pkv_append_decode_attention" if fused else "plain"),
            "block_size": spec.block_size,
            "kv_dtype": f"{quant} codes + fp32 row scales" if quant else spec.dtype,
            "num_seqs": S, "q_heads": Hq, "kv_heads": spec.num_kv_heads,
            "context_tokens": int(st.context_lens.sum()),
            "step_us": round(step_ms * 1000, 2),
            "step_gbs": round(total / (step_ms / 1000) / 1e9, 1),
            "step_frac_of_measured": round(total / (step_ms / 1000) / 1e9 / peak, 4),
            "decode_us": round(dec_ms * 1000, 2),
            "algorithmic_bytes": decode_bytes, "unique_bytes": uniq,
            "decode_frac_of_measured": round(uniq / (dec_ms / 1000) / 1e9 / peak, 4),
            "max_abs_err_vs_oracle": err, "tol": TOL[spec.dtype],
            "parity": "pass" if err <= TOL[spec.dtype] else "FAIL",
            "oracle_s": round(oracle_s, 2),
            "l2": "inputs fit in L2 (launch-bound)" if idx == 0 else "inputs > L2",
        })
        del vals, h, pools, out, ws, app, dec, ref
        torch.cuda.empty_cache()
    return res


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
    if args.suffix_hi is not None:
        from dataclasses import replace
        spec = replace(spec, suffix_hi=args.suffix_hi)
    st = W.make_structure(spec, args.seed)
    scale = 1.0 / math.sqrt(spec.head_dim)
    vals = W.make_values(st, args.seed, device=dev)
    cow = st.cow_pairs if st.cow_pairs.numel() else None
    tables = st.block_tables.to(dev)
    lens = st.context_lens.to(dev)
    slots = st.slot_mapping.to(dev)
    S, Hq, D = vals["q"].shape
    # three resident copies of the cache so every step reads a cold L2
    if args.prefix_aware:
        if not spec.shared_prefix:
            raise SystemExit("--prefix-aware needs a workload with a shared prefix")
        # after the step's copy-on-write every sequence but one holds a private
        # copy of the last prefix block, so the group shares the blocks before it
        shared = spec.shared_prefix // spec.block_size - (1 if cow is not None else 0)
        base = PoolsPrefix(vals["k_pool"], vals["v_pool"], shared)
        copies = [base] + [base.clone() for _ in range(args.copies - 1)]
    elif args.flat:
        if cow is not None:
            raise SystemExit("--flat: flat spans share no blocks (no copy-on-write workloads)")
        if args.kv_quant:
            raise SystemExit("--flat and --kv-quant are separate paths")
        copies = [PoolsFlat.fill(st, vals, dev) for _ in range(args.copies)]
        del vals["k_pool"], vals["v_pool"]      # the rows are in the flat spans now
    else:
        base = PoolsQ.fill(args.kv_quant, st, vals, dev) if args.kv_quant else \
            Pools16(vals["k_pool"], vals["v_pool"], fused=not args.separate_append)
        if args.kv_quant:
            del vals["k_pool"], vals["v_pool"]      # the activations are in the 8-bit cache now
        copies = [base] + [base.clone() for _ in range(args.copies - 1)]
    outs = [torch.empty(S, Hq, D, dtype=vals["q"].dtype, device=dev) for _ in copies]
    wss = [c.workspace(Hq) for c in copies]
    row_bytes = cache_row_bytes(spec, args.kv_quant)
    fused = isinstance(copies[0], Pools16) and copies[0].fused and not args.prefix_aware
    decode_bytes, append_bytes = step_bytes(st, spec, row_bytes, fused=fused)
    total_bytes = decode_bytes + append_bytes
    if cow is not None:
        total_bytes += cow.shape[0] * 2 * 2 * spec.num_kv_heads * spec.block_size * row_bytes
    # bytes the split-K kernel must bring from HBM: shared blocks once
    hbm_decode_bytes = decode_bytes - (int(st.context_lens.sum()) * 2 * spec.num_kv_heads *
                                       row_bytes) + unique_kv_bytes(st, spec, row_bytes)
    # the split-K kernel's own bytes: with the fused append it also writes the new rows
    kernel_bytes = hbm_decode_bytes + (append_bytes if fused else 0)
    stream = torch.cuda.current_stream()
    # prepared calls: the C-ABI arguments are marshalled once per cache copy
    # without copy-on-write only the appended row (each sequence's last) is
    # written by the kernel before the decode, and the other rows of a cache
    # copy were last written three steps before (the copies are used in turn):
    # the decode may gather them while the append runs (pending_tail); a block
    # copy rewrites whole blocks
    pend = 0 if cow is not None else 1
    calls = [c.prepared(vals["q"], vals["k_new"], vals["v_new"], slots, tables, lens, scale, o, w,
                        consumer=args.consumer, pending_tail=pend)
             for c, o, w in zip(copies, outs, wss)]

    def step(i, evs=None, s=None, aevs=None):
        app, dec = calls[i % len(calls)]
        s = s if s is not None else torch.cuda.current_stream()
        if aevs is not None:
            aevs[0].record(s)
        if cow is not None:      # copy-on-write of the last shared block, then append
            copies[i % len(copies)].cow(cow, s)
        if aevs is not None:
            aevs[1].record(s)
        if app is not None:
            app(s)
        if aevs is not None:
            aevs[2].record(s)
        dec(s, timing_events=evs)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if binding.get_error() != 0:
        raise RuntimeError("device error word set during warm-up")

    if args.launch == "graph":
        # each step replays a captured graph of the same kernel launches
        def capture(i):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, capture_error_mode="thread_local"):
                step(i)
            return g
        graphs = [capture(c) for c in range(len(calls))]
        torch.cuda.synchronize()
        for i in range(3):
            graphs[i % len(graphs)].replay()
        torch.cuda.synchronize()

        def run_step(i):
            graphs[i % len(graphs)].replay()
    else:
        def run_step(i):
            step(i)

    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.15)

    # ---- the headline: exactly the step's launches, nothing between them.
    # A device-side sleep ahead of the start event keeps the GPU busy while
    # the host enqueues the first steps, so the timed region begins with work
    # queued (otherwise the host's enqueue of the first launches, ~20 us each,
    # lands inside it); the sleep itself is before the start event.
    barrier(world)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    epoch0 = time.time()
    torch.cuda._sleep(QUEUE_FILL_CYCLES)
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
    if binding.get_error() != 0:
        raise RuntimeError("device error word set during the timed region")

    # ---- per-kernel durations: a second pass over as many steps, with CUDA
    # events on the launching stream around each kernel (events between the
    # launches stop consecutive kernels from overlapping, which is why this
    # pass is kept apart from the headline loop)
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    for evs5 in kev:
        for e in evs5:
            e.record(stream)            # materialise the CUDA event handle (the library
    torch.cuda.synchronize()            # records the decode's pair itself)
    for i in range(args.steps):
        step(i, evs=kev[i][3:5], aevs=kev[i][0:3])
    torch.cuda.synchronize()
    if binding.get_error() != 0:
        raise RuntimeError("device error word set during the per-kernel pass")
    split_avg = sum(e[3].elapsed_time(e[4]) for e in kev) / len(kev)
    side = {}
    if not fused:
        app_ms = sum(e[1].elapsed_time(e[2]) for e in kev) / len(kev)
        side["append"] = {"avg_us": round(app_ms * 1000, 3), "bytes": append_bytes,
                          "gbs": round(append_bytes / (app_ms / 1000) / 1e9, 2),
                          "note": "K/V rows read + written, slots read; launched alone"}
    if cow is not None:
        es = vals["q"].element_size()
        cp_ms = sum(e[0].elapsed_time(e[1]) for e in kev) / len(kev)
        cp_bytes = cow.shape[0] * 2 * 2 * spec.num_kv_heads * spec.block_size * spec.head_dim * es
        side["block_copy"] = {"avg_us": round(cp_ms * 1000, 3), "bytes": cp_bytes,
                              "gbs": round(cp_bytes / (cp_ms / 1000) / 1e9, 2),
                              "note": "whole K and V blocks read + written"}

    per_step_s = ms_max / 1000.0 / args.steps
    value = job_gbs(total_bytes, args.steps, ms_max / 1000.0, world)
    seq_tok = world * int(st.context_lens.sum()) / per_step_s
    peak, peak_kind = peaks()

    # ------------- roofline of the split-K kernel
    # isolated: CUDA events around each launch (the per-kernel pass); when the
    # step is that one kernel alone (fused append, no copy-on-write), the
    # headline loop times back-to-back launches of it, and the average launch
    # duration there is the loop's time over its launches
    iso_gbs = kernel_bytes / (split_avg / 1000.0) / 1e9
    back_to_back = fused and cow is None
    avg_ms = ms / args.steps if back_to_back else split_avg
    ach = kernel_bytes / (avg_ms / 1000.0) / 1e9
    roofline = {"bound": "hbm", "kernel": "decode_split_kernel",
                "achieved": round(ach, 2), "peak": peak, "unit": "GB/s",
                "frac": round(ach / peak, 4),
                "frac_of_nominal": round(ach / NOMINAL_HBM_GBS, 4),
                "traffic": profiled_traffic() if (args.workload == WORKLOAD_INDEX and
                                                  not args.block_size and
                                                  not args.kv_quant and fused) else None,
                "algorithmic_bytes_per_launch": kernel_bytes,
                "logical_bytes_per_launch": decode_bytes + (append_bytes if fused else 0),
                "avg_launch_ms": round(avg_ms, 5),
                "duration": ("timed region / launches: the step is this kernel alone, launched "
                             "back to back with programmatic dependent launch"
                             if back_to_back else
                             "CUDA events around each launch (per-kernel pass)"),
                "isolated": {"avg_launch_ms": round(split_avg, 5), "achieved": round(iso_gbs, 2),
                             "frac": round(iso_gbs / peak, 4),
                             "note": "CUDA events around each launch, which keeps consecutive "
                                     "launches from overlapping"},
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"}

    # ------------- end to end: host inputs in, result out, every step
    e2e = run_e2e(args, st, spec, vals, copies, outs, wss, tables, lens, slots, scale, stream,
                  dev, total_bytes, world)

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max / args.steps, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": args.kv_quant or spec.dtype,
        "data": "synthetic (seeded N(0,1) values, random block tables)",
        "config": {**workload_config(spec, st,
                                     pending=not (cow is not None or args.kv_quant or
                                                  args.prefix_aware),
                                     inputs_ready=not args.flat,
                                     fused=fused),
                   **({"decode": "prefix-aware: the shared prefix decoded once per unit of "
                                 "several sharers' heads, each suffix apart, merged by "
                                 "log-sum-exp in the same launch (pkv_decode_attention_prefix)"}
                      if args.prefix_aware else {}),
                   **({"kv_cache": "flat spans: one virtual range per sequence, physical "
                                   "chunks mapped on demand (pkv_flat_*)",
                       "flat_committed_bytes_per_copy": int(copies[0].fc.info().committed_bytes),
                       "kv_bytes_per_copy": int(st.context_lens.sum()) * 2 * spec.num_kv_heads *
                                            row_bytes} if args.flat else {}),
                   **({"kv_cache": f"{args.kv_quant} codes + fp32 row scales "
                                   f"({row_bytes} B per token and kv head for K, same for V); "
                                   f"{spec.dtype} activations; "
                                   + ("tcgen05 kind::f8f6f4 products (codes as E4M3 operands, q "
                                      "and p as three E4M3 parts, fp32 accumulators in TMEM)"
                                      if args.kv_quant == "fp8_e4m3" else
                                      "codes to fp16 in registers, mma.sync")}
                      if args.kv_quant else {}),
                   "l2": f"inputs > L2: the step cycles through {len(copies)} resident copies "
                         f"of the cache ({len(copies)} x {2 * st.num_blocks * spec.num_kv_heads * spec.block_size * row_bytes / 1e9:.2f} GB)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "launch": "CUDA-graph replay of the step's kernel launches (captured through the C ABI)"
                             if args.launch == "graph" else "eager C-ABI calls"},
        "seq_tokens_per_s": round(seq_tok, 1),
        "hbm_frac_of_measured": round(value / peak / world, 4),
        # the same figure against the nominal 8 TB/s of GB300 HBM3e; the 75 %
        # decode-kernel target is judged against the measured copy peak
        "hbm_frac_of_nominal": round(value / NOMINAL_HBM_GBS / world, 4),
        "roofline": roofline,
        "other_kernels": side or None,
        "block_manager": time_block_manager(st, spec) if rank == 0 else None,
        # the fused step is one launch; otherwise append + decode (the
        # prefix-aware decode is one launch too); plus the copy-on-write launch
        "gpu_launches": ((1 if fused else 2) + (1 if cow is not None else 0)) * args.steps,
        "clocks": clocks,
        "wall_s_timed_region": round(wall, 4),
        "host_enqueue_s": round(enqueue_s, 4),
        "e2e": e2e,
    }
    plain = (args.workload == WORKLOAD_INDEX and not (args.block_size or args.dtype or
                                                        args.kv_quant or args.flat or
                                                        args.prefix_aware or args.suffix_hi))
    if rank == 0 and plain and not args.no_workloads:
        line["workloads"] = workload_sweep(args, dev, peak)
    if rank == 0 and not args.no_cpu_baseline:
        from oracle import oracle
        h = host_inputs_from_generator(st, args.seed, dev, args.kv_quant)
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


def _packed(tensors, dev):
    """One pinned host byte buffer holding `tensors` back to back (16-byte
    aligned), a device byte buffer of the same size, and views of the device
    buffer with each tensor's dtype and shape: one copy moves a step's inputs."""
    offs, n = [], 0
    for t in tensors:
        offs.append(n)
        n += (t.numel() * t.element_size() + 15) // 16 * 16
    host = torch.zeros(n, dtype=torch.uint8).pin_memory()
    for t, o in zip(tensors, offs):
        b = t.numel() * t.element_size()
        host[o:o + b].copy_(t.detach().cpu().contiguous().view(-1).view(torch.uint8))
    dbuf = torch.empty(n, dtype=torch.uint8, device=dev)
    views = [dbuf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
             for t, o in zip(tensors, offs)]
    return host, dbuf, views


def run_e2e(args, st, spec, vals, copies, outs, wss, tables, lens, slots, scale, stream, dev,
            total_bytes, world):
    """The step through the public API with its inputs (q, the new K/V rows,
    slot mapping, block tables, lengths) copied from pinned host memory in one
    transfer and its output read back to pinned host memory, every step.
    Serial: copy in, append + decode, copy out, wait, per step. Pipelined (the
    reported value): two steps in flight, the input and output copies each on
    a stream of their own; step i's inputs land in one of two device buffers
    while step i - 1 computes, and the host waits for step i - 1's output
    before it enqueues step i + 1."""
    from paged_kv_cache_47_gb300 import binding
    inputs = [vals["q"], vals["k_new"], vals["v_new"], st.block_tables, st.context_lens,
              st.slot_mapping]
    h_in, d_in0, v0 = _packed(inputs, dev)
    _, d_in1, v1 = _packed(inputs, dev)
    sets = [v0, v1]
    bufs = [d_in0, d_in1]
    h_out = [torch.empty(vals["q"].shape, dtype=vals["q"].dtype).pin_memory() for _ in range(2)]
    h2d = h_in.numel()
    d2h = h_out[0].numel() * h_out[0].element_size()
    steps = min(args.steps, args.e2e_steps)
    cow = st.cow_pairs if st.cow_pairs.numel() else None
    # prepared calls per (input set, workload copy)
    pend = 0 if cow is not None else 1
    calls = [[(*c.prepared(v[0], v[1], v[2], v[5], v[3], v[4], scale, out, ws,
                           pending_tail=pend), out)
              for c, out, ws in zip(copies, outs, wss)] for v in sets]

    def compute(i, b):
        app, dec, out = calls[b][i % len(copies)]
        if cow is not None:
            copies[i % len(copies)].cow(cow, stream)
        if app is not None:
            app(stream)
        dec(stream)
        return out

    def serial(i):
        bufs[0].copy_(h_in, non_blocking=True)
        out = compute(i, 0)
        h_out[0].copy_(out, non_blocking=True)
        stream.synchronize()            # the step's result is on the host

    in_s, out_s = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    # The pipelined loop drives the copies and the cross-stream order through
    # the CUDA runtime directly (resolved through libpkv's own dependency on
    # it), as a C++ serving loop would: torch's per-call overhead would
    # otherwise bound the loop on the host.
    rt = binding.lib()
    vp, sz = ctypes.c_void_p, ctypes.c_size_t
    rt.cudaMemcpyAsync.argtypes = [vp, vp, sz, ctypes.c_int, vp]
    rt.cudaEventCreateWithFlags.argtypes = [ctypes.POINTER(vp), ctypes.c_uint]
    rt.cudaEventRecord.argtypes = [vp, vp]
    rt.cudaStreamWaitEvent.argtypes = [vp, vp, ctypes.c_uint]
    rt.cudaEventSynchronize.argtypes = [vp]
    rt.cudaEventDestroy.argtypes = [vp]

    def event():
        e = vp()
        if rt.cudaEventCreateWithFlags(ctypes.byref(e), 2) != 0:   # cudaEventDisableTiming
            raise RuntimeError("cudaEventCreateWithFlags failed")
        return e

    ev_in, ev_dec, ev_out = [event(), event()], [event(), event()], [event(), event()]
    s_comp, s_in, s_out = (vp(stream.cuda_stream), vp(in_s.cuda_stream), vp(out_s.cuda_stream))
    h_in_p = vp(h_in.data_ptr())
    bufs_p = [vp(b.data_ptr()) for b in bufs]
    h_out_p = [vp(h.data_ptr()) for h in h_out]
    outs_p = [vp(o.data_ptr()) for o in outs]
    H2D, D2H = 1, 2

    def pipelined(n):
        for i in range(n):
            b = i % 2
            if i >= 2:
                rt.cudaStreamWaitEvent(s_in, ev_dec[b], 0)   # step i - 2 is done with buffer b
            rt.cudaMemcpyAsync(bufs_p[b], h_in_p, h2d, H2D, s_in)
            rt.cudaEventRecord(ev_in[b], s_in)
            rt.cudaStreamWaitEvent(s_comp, ev_in[b], 0)
            compute(i, b)
            rt.cudaEventRecord(ev_dec[b], s_comp)
            rt.cudaStreamWaitEvent(s_out, ev_dec[b], 0)
            rt.cudaMemcpyAsync(h_out_p[b], outs_p[i % len(copies)], d2h, D2H, s_out)
            rt.cudaEventRecord(ev_out[b], s_out)
            if i >= 1:
                rt.cudaEventSynchronize(ev_out[(i - 1) % 2])   # step i - 1's result is on the host
        rt.cudaEventSynchronize(ev_out[(n - 1) % 2])

    def timed(fn):
        barrier(world)
        t0 = time.perf_counter()
        fn()
        dt = time.perf_counter() - t0
        return reduce_max(dt, world, dev)

    for i in range(3):
        serial(i)
    dt_serial = timed(lambda: [serial(i) for i in range(steps)])
    pipelined(3)
    dt = timed(lambda: pipelined(steps))
    for e in ev_in + ev_dec + ev_out:
        rt.cudaEventDestroy(e)
    gbs = lambda t: round(world * total_bytes * steps / t / 1e9, 2)  # noqa: E731
    return {"value": gbs(dt), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": steps, "ms_per_step": round(1000 * dt / steps, 4),
            "mode": "pipelined: one H2D of the packed inputs and one D2H of the output per "
                    "step, each on a copy stream of its own, two steps in flight; copies "
                    "and stream order through the CUDA runtime directly",
            "serial": {"value": gbs(dt_serial), "ms_per_step": round(1000 * dt_serial / steps, 4),
                       "mode": "copy in, step, copy out, wait, one step at a time"}}


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
    ap.add_argument("--prefix-aware", action="store_true",
                    help="decode shared prefixes once per group of sharers (shared-prefix workload)")
    ap.add_argument("--suffix-hi", type=int, default=None,
                    help="override the shared-prefix workload's largest private suffix")
    ap.add_argument("--flat", action="store_true",
                    help="flat per-sequence spans in virtual memory instead of a paged pool")
    ap.add_argument("--kv-quant", choices=["int8", "fp8_e4m3"], default=None,
                    help="8-bit KV cache (codes + fp32 row scales) instead of the workload's dtype")
    ap.add_argument("--consumer", type=int, default=0,
                    help="math path: 0 auto, 1 CUDA cores, 2 tensor cores (16-bit only)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--separate-append", action="store_true",
                    help="16-bit paged step as pkv_append + pkv_decode_attention (two launches) "
                         "instead of pkv_append_decode_attention")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the other workloads' figures in the default line")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
