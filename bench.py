#!/usr/bin/env python3
"""Benchmark of the kvx hot path on one GB300 (or N replicas under torchrun).

One step = one decode step of the Qwen3-4B-shaped workload: for each of its 36
layers, split decode attention over that layer's head-group paged KV cache
(the log-sum-exp merge of split heads runs in the same launch). The other
decode workloads (the 32k-context step, the Qwen2.5-32B step, the Llama-3-8B
sparse step and the tiny fp32 case) are timed the same way and reported under
`workloads`; the KV-RM gather (256 sequences, fragmented 40 GB pool,
fixed-shape staging) is timed in its own loop. All in one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line on rank 0. `--impl reference` times the fp64 CPU oracle
on the host cores on a bounded sample of the same workload.
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

import synth  # noqa: E402

METRIC = "decode-attn KV GB/s and % of GB300 HBM roofline; gather GB/s"
FALLBACK_HBM = 6800.0
EXTRA_WORKLOADS = ["qwen3_4b_32k", "qwen25_32b", "llama3_sparse", "tiny"]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="qwen3_4b",
                    choices=["qwen3_4b", "qwen3_4b_32k", "qwen25_32b", "llama3_sparse"])
    ap.add_argument("--no-gather", action="store_true")
    ap.add_argument("--no-frame", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-group-sweep", action="store_true")
    ap.add_argument("--no-sparse", action="store_true")
    ap.add_argument("--no-workloads", action="store_true")
    ap.add_argument("--layers", type=int, default=0,
                    help="decode only the first N layers of the workload (profiling "
                         "captures); 0 = all")
    ap.add_argument("--cpu-seconds", type=float, default=3.0,
                    help="oracle time per workload in the CPU baseline")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM, "fallback"


KERNEL_SOURCES = ["attn_mma.cu", "ptx.cuh", "split_merge.cuh", "kvx_internal.h", "abi.cpp",
                  "plan.cpp"]
PROFILE = os.path.join(ROOT, "profiles", "attn_mma_qwen3_4b.json")


def kernel_source_hash() -> str:
    """sha256 over the attention kernel's source files, to tell whether a
    committed ncu capture still describes the kernel that runs."""
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "paged_non_uniform_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def profiled_traffic():
    """(dram bytes per launch, algorithmic bytes of that launch) from the
    committed ncu figures, or None if the kernel has changed since."""
    try:
        with open(PROFILE) as f:
            d = json.load(f)
        if d.get("kernel_source_sha256") != kernel_source_hash():
            return None
        return float(d["dram_bytes_per_launch"]), float(d["algorithmic_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


def describe(cfg) -> str:
    return (f"{cfg.name} decode: {cfg.layers} layers, batch {cfg.B}, {cfg.Hq} q / {cfg.Hkv} KV "
            f"heads, head_dim {cfg.D}, {cfg.dtype}, page {cfg.P}, {cfg.num_groups} head groups, "
            f"seq_len {int(cfg.seq_len.min())}..{int(cfg.seq_len.max())}, "
            f"kept tokens/step {int(cfg.n.sum())}")


def config_of(cfg) -> dict:
    """The `config` object of the JSON line (the same for both arms)."""
    return {"workload": describe(cfg),
            "l2": "inputs larger than L2: each step streams "
                  f"{cfg.kv_bytes_step() / 1e9:.1f} GB of distinct KV pages",
            "plan": "balanced ahead-of-time split, two persistent blocks per SM",
            "step": "one replay of a CUDA graph holding the step's kvx_decode_attn launches "
                    "(one per layer, captured from the C-ABI calls)",
            "early_kv": "on: each launch's load warps fill their rings before the previous "
                        "launch completes, which writes no page or page table"}


# ------------------------------------------------------------ CPU oracle
def host_group_pages(cfg, layer):
    """Pages each group needs (ceil of the group's longest head / P), as the
    library reports them; used to rebuild the GPU arm's page tables."""
    hg = cfg.head_group[layer]
    gp = np.zeros((cfg.num_groups, cfg.B), dtype=np.int64)
    for h in range(cfg.Hkv):
        gp[hg[h]] = np.maximum(gp[hg[h]], (cfg.n[layer][:, h] + cfg.P - 1) // cfg.P)
    return gp


def host_batch(cfg, layer=0, b0=0, max_rows=1 << 20, table_seed=11):
    """The oracle's inputs for sequences b0..b1-1 of one layer, rebuilt on the
    host from the seeded value table and page tables the GPU arm uses
    (synth.device.TableLayer with seed 0): q [nb][Hq][D], dense k and v
    [nb][Hkv][nmax][D] holding each head's kept rows at positions 0..n-1,
    lengths, kept sets, and the KV bytes (storage type) they stand for. As
    many sequences as fit in max_rows rows per tensor (at least one)."""
    from synth.device import page_tables_for, rows_in_group
    table_rows = 1 << 19
    vals = synth.value_table(table_seed, table_rows * cfg.D, cfg.dtype)
    vals = (synth.bf16_bits_to_f32(vals) if cfg.dtype == "bf16" else vals).reshape(table_rows,
                                                                                   cfg.D)
    n = cfg.n[layer]
    b1 = b0 + 1
    while b1 < cfg.B and (b1 + 1 - b0) * cfg.Hkv * int(n[b0:b1 + 1].max()) <= max_rows:
        b1 += 1
    tables, _ = page_tables_for(host_group_pages(cfg, layer), 0 * 131 + layer, 0)
    hg = cfg.head_group[layer]
    rows, gsize = rows_in_group(hg), np.bincount(hg, minlength=cfg.num_groups)
    gen = synth.rng(0 * 1009 + layer)
    sh = gen.integers(0, table_rows, size=(cfg.num_groups, 2)).astype(np.int64)
    q = synth.normal(gen, (cfg.B, cfg.Hq, cfg.D), cfg.dtype)
    nmax = int(n[b0:b1].max())
    k = np.zeros((b1 - b0, cfg.Hkv, nmax, cfg.D))
    v = np.zeros_like(k)
    kept = []
    for b in range(b0, b1):
        for h in range(cfg.Hkv):
            gi = int(hg[h])
            t = np.arange(int(n[b, h]), dtype=np.int64)
            ids = (tables[gi][b, t // cfg.P].astype(np.int64) * int(gsize[gi]) +
                   int(rows[h])) * cfg.P + t % cfg.P
            k[b - b0, h, :t.size] = vals[(sh[gi, 0] + ids) % table_rows]
            v[b - b0, h, :t.size] = vals[(sh[gi, 1] + ids) % table_rows]
            kept.append(np.arange(t.size, dtype=np.int32))
    es = 2 if cfg.dtype == "bf16" else 4
    nbytes = int(n[b0:b1].sum()) * 2 * cfg.D * es
    qb = np.ascontiguousarray(q[b0:b1], dtype=np.float64)
    return (qb, k, v, np.full(b1 - b0, nmax, np.int32), kept), nbytes, b1 - b0


def oracle_timing(cfg, seconds):
    """Times oracle_decode_attn, as it stands, on one batch of the workload's
    layer-0 sequences (OpenMP over the batch's (sequence, KV head) pairs),
    repeated until `seconds` of oracle time. Returns (GB/s of KV, threads
    used, description)."""
    import oracle
    orc = oracle.load()
    args, nbytes, nseq = host_batch(cfg)
    scale = 1.0 / math.sqrt(cfg.D)
    spent, reps = 0.0, 0
    while spent < seconds or reps == 0:
        t0 = time.perf_counter()
        orc.decode_attn(*args, scale)
        spent += time.perf_counter() - t0
        reps += 1
    heads = nseq * cfg.Hkv
    cores = min(orc.num_threads(), heads)
    return (nbytes * reps / spent / 1e9, cores,
            f"{nseq} sequences x {cfg.Hkv} KV heads of {cfg.name} layer 0 ({nbytes / 1e9:.3f} "
            f"GB of {cfg.dtype} KV per call), {reps} calls in {spent:.1f} s of fp64 oracle "
            f"time, OpenMP over the {heads} (sequence, KV head) pairs")


def oracle_layer_step(name, rate_gbs):
    """The oracle's time for the whole of layer 0 of a workload at the rate
    it measured on its batch, and the same times the workload's layer count:
    an extrapolation, not a timed step."""
    full = synth.decode_config(name, seed=0)
    layer_s = full.kv_bytes_layer(0) / (rate_gbs * 1e9)
    return {"layer_s": layer_s, "step_s_extrapolated": layer_s * full.layers,
            "layers": full.layers}


def cpu_baseline(cfg, seconds, extra=()):
    value, cores, sample = oracle_timing(cfg, seconds)
    out = {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample,
           **oracle_layer_step(cfg.name, value), "workloads": {}}
    for name in extra:
        c = synth.decode_config(name, seed=0, layers=1)
        v, cr, smp = oracle_timing(c, seconds)
        out["workloads"][name] = {"value": v, "unit": "GB/s", "cores": cr, "sample": smp,
                                  **oracle_layer_step(name, v)}
    return out


def host_cpu() -> dict:
    """CPU model and logical CPU count of the host."""
    model = ""
    try:
        for line in open("/proc/cpuinfo"):
            key = line.split(":", 1)[0].strip().lower()
            if key in ("model name", "cpu part", "hardware"):
                model = line.split(":", 1)[1].strip()
                if key != "model name":
                    model = f"{key} {model}"
                break
    except OSError:
        pass
    return {"model": model or "unknown", "nproc": os.cpu_count()}


def cpu_gather_baseline(S=32, num_phys=65536):
    """The oracle's block-by-block gather (memcpy per block, OpenMP over rows)
    on a sample of the KV-RM workload: S sequences of the same length mix
    over a randomly permuted pool of num_phys 32 KB blocks per tensor (K and
    V), timed on the host cores. Values are irrelevant to a copy; the
    buffers are touched before timing."""
    import oracle
    orc = oracle.load()
    cfg = synth.gather_config(seed=0, S=S, num_phys=num_phys)
    moved, secs = 0, 0.0
    for _ in range(2):  # K and V
        pool = np.empty((cfg.num_phys, cfg.block_bytes), np.uint8)
        pool.fill(1)
        staging = np.empty((cfg.S, cfg.row_bytes), np.uint8)
        staging.fill(0)
        t0 = time.perf_counter()
        orc.gather(cfg.bt, cfg.nb, pool, staging)
        secs += time.perf_counter() - t0
        moved += 2 * int(cfg.nb.sum()) * cfg.block_bytes
    return {"value": moved / secs / 1e9, "unit": "GB/s moved (read+write)",
            "cores": orc.num_threads(), "kind": "oracle",
            "sample": f"{S} sequences, {int(cfg.nb.sum())} live 32 KB blocks per tensor, K and V "
                      f"pools of {num_phys} blocks each ({moved / 1e9:.2f} GB moved)"}


def copy_ceiling(dev, stream, torch, gib=4, reps=10) -> float:
    """Practical ceiling: device-to-device copy of a buffer larger than L2 with
    the CUDA runtime (cudaMemcpyAsync through torch), GB/s read + write."""
    a = torch.empty(gib << 30, dtype=torch.uint8, device=dev)
    b = torch.empty_like(a)
    a.fill_(1)
    for _ in range(2):
        b.copy_(a)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        b.copy_(a)
    e1.record(stream)
    torch.cuda.synchronize()
    gbs = 2 * (gib << 30) * reps / (e0.elapsed_time(e1) * 1e-3) / 1e9
    del a, b
    torch.cuda.empty_cache()
    return gbs


def run_reference(args, rank, world):
    """The oracle as it stands, on the host cores: each step runs it over the
    same bounded sample of the workload (the first sequences of layer 0, one
    call with OpenMP over all their (sequence, KV head) pairs), repeated so
    that warm-up plus timed steps take about half a minute."""
    import oracle
    if rank != 0:
        return
    cfg = synth.decode_config(args.workload, seed=0)
    orc = oracle.load()
    total_steps = max(args.steps + args.warmup, 1)
    target = max(0.02, 30.0 / total_steps)
    call, nbytes, nseq = host_batch(cfg)
    scale = 1.0 / math.sqrt(cfg.D)
    t0 = time.perf_counter()
    orc.decode_attn(*call, scale)
    reps = max(1, int(round(target / max(time.perf_counter() - t0, 1e-6))))
    secs = []
    for i in range(total_steps):
        t0 = time.perf_counter()
        for _ in range(reps):
            orc.decode_attn(*call, scale)
        if i >= args.warmup:
            secs.append(time.perf_counter() - t0)
    sec = sum(secs)
    value = nbytes * reps * len(secs) / sec / 1e9
    cores = min(orc.num_threads(), nseq * cfg.Hkv)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * sec / max(len(secs), 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(cfg),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": f"each step: the fp64 oracle over the first {nseq} "
                                       f"sequences of layer 0 ({nbytes / 1e9:.3f} GB of bf16 "
                                       f"KV), {reps} times, OpenMP over their "
                                       f"{nseq * cfg.Hkv} (sequence, KV head) pairs",
                             "host": host_cpu()},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- replicas
def rank_seed(rank: int) -> int:
    """Seed of the batch a replica serves: every rank decodes its own batch."""
    return rank


def max_over_ranks(ms: float, dist, device=None) -> float:
    """The slowest rank's time (the whole job finishes when it does)."""
    if dist is None:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, dist, device=None) -> float:
    """Units all ranks processed (each rank's batch differs)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def job_rate(total_bytes: float, ms: float) -> float:
    """Whole-job GB/s: bytes all ranks processed over the slowest rank's time."""
    return total_bytes / (ms * 1e-3) / 1e9


# ------------------------------------------------------------------ clocks
class Clocks:
    def __init__(self):
        self.proc = None
        self.path = os.environ.get("KVX_BENCH_CLOCKS") or os.path.join(
            tempfile.gettempdir(), "kvx_bench_clocks.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                 "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                 "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
            dev = os.environ.get("CUDA_VISIBLE_DEVICES", "0").split(",")[0] or "0"
            self.proc = subprocess.Popen(["nvidia-smi", "-i", dev, f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "samples": len(sm), "reasons": sorted(reasons)}


# -------------------------------------------------------------- GPU arm
class DecodeSetup:
    """Plans (balanced, default block count) and head-group pools of every
    layer of one decode workload, filled on the GPU from a seeded value
    table; one shared workspace and an output per layer."""

    def __init__(self, cfg, table, dev, kvx, torch):
        from synth.device import TableLayer
        self.cfg, self.kvx = cfg, kvx
        dtype = kvx.KVX_BF16 if cfg.dtype == "bf16" else kvx.KVX_F32
        self.plans, self.layers, self.plan_us = [], [], []
        for l in range(cfg.layers):
            p = kvx.kvx_plan_create(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, cfg.P, cfg.num_groups, dtype,
                                    cfg.budget[l], cfg.seq_len, cfg.head_group[l], 0)
            kvx.kvx_plan_upload(p)
            # the step's kernels are these attention launches, and none of them
            # writes pages or page tables: the load warps may start before the
            # previous layer's launch has completed (kvx_plan_set_early_kv)
            p.set_early_kv(True)
            self.plan_us.append(p.stats()["plan_us"])
            self.plans.append(p)
            self.layers.append(TableLayer(cfg, l, table, p.group_pages(), seed=0, device=dev))
        ws_bytes = max(p.workspace_bytes() for p in self.plans)
        self.ws = torch.zeros(max(ws_bytes, 256) // 4 + 64, dtype=torch.int32, device=dev)
        self.outs = torch.empty((cfg.layers, cfg.B, cfg.Hq, cfg.D), dtype=torch.float32,
                                device=dev)
        self.bytes_layer = [cfg.kv_bytes_layer(l) for l in range(cfg.layers)]
        self.bytes_step = sum(self.bytes_layer)
        self.graph = None

    def call(self, l, stream, q=None, out=None):
        lay = self.layers[l]
        self.kvx.kvx_decode_attn(self.plans[l], lay.q if q is None else q, lay.k_pools,
                                 lay.v_pools, lay.pool_pages, lay.pt, lay.strides, lay.budget,
                                 lay.seq_len, 0.0, self.outs[l] if out is None else out, self.ws,
                                 stream=stream)

    def step(self, stream):
        if self.graph is not None:
            self.graph.replay()
            return
        for l in range(self.cfg.layers):
            self.call(l, stream)

    def capture(self, torch):
        """Captures the step's per-layer kvx_decode_attn calls in one CUDA
        graph (after direct calls have set up every kernel instance); step()
        then replays it on the current stream. Decode steps launch one short
        kernel per layer; replaying the captured launches keeps the host's
        per-call argument handling out of the step, so the kernels run back to
        back with their programmatic dependent launches overlapping."""
        self.graph = None
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            st = torch.cuda.current_stream()
            for l in range(self.cfg.layers):
                self.call(l, st)
        torch.cuda.synchronize()
        self.graph = g

    def status(self) -> int:
        return self.kvx.kvx_workspace_status(self.ws)

    def per_launch(self, stream, torch, steps):
        """A second pass of `steps` steps with a CUDA event after every launch
        (which serialises the programmatic dependent launches): the rate of
        each launch on its own, GB/s mean and p10/p50/p90, and its mean
        duration."""
        L = self.cfg.layers
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(L + 1)] for _ in range(steps)]
        for s in range(steps):
            ev[s][0].record(stream)
            for l in range(L):
                self.call(l, stream)
                ev[s][l + 1].record(stream)
        torch.cuda.synchronize()
        call_ms = np.array([[ev[s][l].elapsed_time(ev[s][l + 1]) for l in range(L)]
                            for s in range(steps)])
        rates = np.array([[self.bytes_layer[l] / (call_ms[s, l] * 1e-3) for l in range(L)]
                          for s in range(steps)]).reshape(-1) / 1e9
        return {"mean_gbs": float(rates.mean()),
                "p10_gbs": float(np.percentile(rates, 10)),
                "p50_gbs": float(np.percentile(rates, 50)),
                "p90_gbs": float(np.percentile(rates, 90)),
                "mean_call_us": float(call_ms.mean() * 1e3)}


def timed_steps(setup, stream, torch, steps, warmup, dist=None, dev=None, clocks=None):
    """W untimed steps, then exactly K steps between two events on the
    launching stream (barrier and synchronize on both sides); a step is one
    replay of the captured step graph. Returns (ms per step as the max over
    ranks, clock record or None)."""
    setup.step(stream)  # direct calls: every kernel instance is set up
    torch.cuda.synchronize()
    setup.capture(torch)
    for _ in range(warmup):
        setup.step(stream)
    torch.cuda.synchronize()
    assert setup.status() == 0, "device status set during warm-up"
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    if clocks:
        clocks.start()
        time.sleep(0.3)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(steps):
        setup.step(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop() if clocks else None
    if dist:
        dist.barrier()
    assert setup.status() == 0, "device status set during the timed region"
    return max_over_ranks(t0.elapsed_time(t1) / steps, dist, dev), clk


def workload_line(setup, ms_step, peak, per_launch, note):
    cfg = setup.cfg
    value = setup.bytes_step / (ms_step * 1e-3) / 1e9
    return {"workload": describe(cfg), "value": value, "unit": "GB/s", "frac": value / peak,
            "ms_per_step": ms_step, "kv_bytes_per_step": setup.bytes_step,
            "seq_heads_per_s": cfg.B * cfg.Hq * cfg.layers / (ms_step * 1e-3),
            "launches_per_step": cfg.layers, "per_launch": per_launch,
            "plan_host_us_per_layer": float(np.mean(setup.plan_us)), "l2": note}


def bench_workload(name, table_for, dev, stream, peak, steps, warmup, kvx, torch):
    """One extra decode workload in its own pools, freed afterwards."""
    cfg = synth.decode_config(name, seed=0)
    setup = DecodeSetup(cfg, table_for(cfg), dev, kvx, torch)
    if name == "tiny":
        # One layer of 90.6 KB: each timed call follows an L2 flush (a write
        # of a buffer larger than L2), with events around the call alone.
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        setup.step(stream)
        setup.capture(torch)
        for _ in range(warmup):
            setup.step(stream)
        ms = []
        for _ in range(steps):
            flush.zero_()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            setup.step(stream)
            b.record(stream)
            b.synchronize()
            ms.append(a.elapsed_time(b))
        assert setup.status() == 0
        line = workload_line(setup, float(np.mean(ms)), peak, None,
                             "each call after an L2 flush (256 MiB write); events around the "
                             "call; fp32 K/V, CUDA-core kernel; launch-bound")
        del flush
    else:
        ms, _ = timed_steps(setup, stream, torch, steps, warmup)
        line = workload_line(setup, ms, peak, setup.per_launch(stream, torch, max(3, steps // 4)),
                             f"inputs larger than L2: {setup.bytes_step / 1e9:.2f} GB of "
                             "distinct KV pages per step")
    del setup
    torch.cuda.empty_cache()
    return line


def run_ours(args, rank, world):
    import torch
    from paged_non_uniform_gb300 import build
    build.build()
    from paged_non_uniform_gb300 import kvx
    from synth.device import ValueTable

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    stream = torch.cuda.current_stream()
    peak, peak_kind = peaks()

    cfg = synth.decode_config(args.workload, seed=rank_seed(rank), layers=args.layers or None)
    tables = {}

    def table_for(c):
        key = (c.dtype, c.D)
        if key not in tables:
            tables[key] = ValueTable(seed=11 + rank_seed(rank), rows=1 << 19, D=c.D,
                                     dtype=c.dtype, device=dev)
        return tables[key]

    sms = kvx.kvx_device_sm_count()
    setup = DecodeSetup(cfg, table_for(cfg), dev, kvx, torch)
    bytes_step = setup.bytes_step

    # ---- timed region: K whole steps between two events
    ms_step, clk = timed_steps(setup, stream, torch, args.steps, args.warmup, dist, dev, Clocks())
    bytes_job = sum_over_ranks(bytes_step, dist, dev)
    value = job_rate(bytes_job, ms_step)

    # ---- roofline of the attention kernel. The step launches nothing but
    # this kernel, one launch per layer, so its mean duration inside the timed
    # region is the step time over the launches; achieved = algorithmic KV
    # bytes of the mean launch over that duration.
    launches_per_step = cfg.layers
    in_step_us = ms_step * 1e3 / launches_per_step
    achieved = float(np.mean(setup.bytes_layer)) / (in_step_us * 1e-6) / 1e9
    per_launch = setup.per_launch(stream, torch, args.steps)
    prof = profiled_traffic()
    # ncu traffic of the profiled launch (layer 0), scaled to the mean launch
    traffic = (prof[0] * np.mean(setup.bytes_layer) / prof[1]) if prof else None

    # ---- load balance of layer 0 under the three plans (same kernel)
    balance = (measure_balance(cfg, setup.layers[0], setup.ws, stream, kvx, torch)
               if rank == 0 else None)

    # ---- end to end through the public API with host buffers
    e2e = end_to_end(setup, dev, stream, dist, bytes_job, args.steps, torch)
    plan_us = float(np.mean(setup.plan_us))

    del setup
    torch.cuda.empty_cache()

    # ---- the other decode workloads, each in its own pools
    workloads = None
    if rank == 0 and not args.no_workloads:
        workloads = {}
        for name in EXTRA_WORKLOADS:
            if name != args.workload:
                workloads[name] = bench_workload(name, table_for, dev, stream, peak, args.steps,
                                                 args.warmup, kvx, torch)

    # ---- head-group size sweep (first layers of the same workload)
    gsweep = None
    if rank == 0 and not args.no_group_sweep:
        gsweep = group_sweep(cfg, table_for(cfg), dev, stream, peak, kvx, torch)

    sparse = None
    if rank == 0 and not args.no_sparse:
        sparse = sparse_select(dev, stream, peak, kvx, torch)

    # ---- gather (KV-RM movement workload)
    gather = None
    if not args.no_gather:
        tables.clear()
        torch.cuda.empty_cache()
        gather = bench_gather(args, dev, stream, peak, dist, world, rank)

    cpu = None
    ceiling = copy_ceiling(dev, stream, torch)
    if rank == 0 and not args.no_cpu:
        cpu = cpu_baseline(cfg, args.cpu_seconds,
                           [w for w in ("qwen25_32b", "llama3_sparse", "tiny")
                            if w != args.workload])
        cpu["host"] = host_cpu()
        cpu["gather"] = cpu_gather_baseline()

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) bf16 K/V, fragmented page tables)",
            "config": config_of(cfg), "sms": sms,
            "frac_of_hbm": value / world / peak,
            "seq_heads_per_s": world * cfg.B * cfg.Hq * cfg.layers / (ms_step * 1e-3),
            "kv_bytes_per_step": bytes_job,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "traffic_note": "ncu dram read+write of the profiled layer-0 launch, "
                                         "scaled to the mean launch by algorithmic bytes"
                                         if prof else "kernel changed since the committed "
                                                      "capture",
                         "kernel": "attn_mma_kernel<128> (one launch per layer call; the only "
                                   "kernel of the step)",
                         "timing": "in-step: frac and achieved use the mean launch duration "
                                   "inside the timed region (step time / launches per step)",
                         "in_step_launch_us": in_step_us,
                         "per_launch_events": dict(per_launch, frac=per_launch["mean_gbs"] / peak,
                                                   timing="second pass of K steps with an "
                                                          "event after every launch, which "
                                                          "serialises the programmatic "
                                                          "dependent launches"),
                         "peak_source": f"{peak_kind} hbm_gbs", "copy_ceiling_gbs": ceiling},
            "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk,
            "plan_host_us_per_layer": plan_us,
            "workloads": workloads,
            "gather": gather,
            "balance": balance,
            "group_sweep": gsweep,
            "sparse_select": sparse,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def end_to_end(setup, dev, stream, dist, bytes_job, steps, torch):
    """The same step through the public API with host buffers: every step
    copies its q from pinned host memory and reads its outputs back. The
    copies run on a second stream, double-buffered: step k+1's q goes up and
    step k-1's outputs come down while step k computes."""
    cfg = setup.cfg
    q_host = torch.empty((cfg.layers, cfg.B, cfg.Hq, cfg.D), dtype=torch.bfloat16,
                         pin_memory=True)
    for l in range(cfg.layers):
        q_host[l].copy_(setup.layers[l].q.cpu())
    e2e_steps = max(3, steps // 2)
    q_dev = [torch.empty_like(q_host, device=dev) for _ in range(2)]
    out_dev = [torch.empty_like(setup.outs) for _ in range(2)]
    out_host = [torch.empty(tuple(setup.outs.shape), dtype=torch.float32, pin_memory=True)
                for _ in range(2)]
    copy_stream = torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]    # q of buffer i is on the device
    ev_done = [torch.cuda.Event() for _ in range(2)]  # compute on buffer i has finished
    ev_out = [torch.cuda.Event() for _ in range(2)]   # outputs of buffer i are on the host

    def stage_in(i):
        copy_stream.wait_event(ev_done[i])
        with torch.cuda.stream(copy_stream):
            q_dev[i].copy_(q_host, non_blocking=True)
        ev_in[i].record(copy_stream)

    def e2e_step(k):
        i = k % 2
        stage_in(1 - i)                  # next step's q, behind step k-1's compute
        stream.wait_event(ev_in[i])
        stream.wait_event(ev_out[i])     # step k-2's outputs have left out_dev[i]
        for l in range(cfg.layers):
            setup.call(l, stream, q=q_dev[i][l], out=out_dev[i][l])
        ev_done[i].record(stream)
        copy_stream.wait_event(ev_done[i])
        with torch.cuda.stream(copy_stream):
            out_host[i].copy_(out_dev[i], non_blocking=True)
        ev_out[i].record(copy_stream)

    stage_in(0)
    for k in range(2):
        e2e_step(k)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    h0 = time.perf_counter()
    stage_in(0)
    for k in range(e2e_steps):
        e2e_step(k)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks((time.perf_counter() - h0) * 1e3 / e2e_steps, dist, dev)
    return {"value": job_rate(bytes_job, e2e_ms), "unit": "GB/s",
            "h2d_bytes_per_step": int(q_host.numel() * 2),
            "d2h_bytes_per_step": int(out_host[0].numel() * 4)}


def measure_balance(cfg, lay, ws, stream, kvx, torch):
    """Layer 0 under the balanced ahead-of-time plan and the two naive plans:
    kernel time (median of 20) and the spread of per-block busy times from
    the kernel's own trace (SM id, start, end, tokens per block)."""
    res = {}
    names = {kvx.KVX_PLAN_BALANCED: "balanced_aot", kvx.KVX_PLAN_PER_HEAD: "one_block_per_head",
             kvx.KVX_PLAN_UNIFORM: "uniform_split"}
    out = torch.empty((cfg.B, cfg.Hq, cfg.D), dtype=torch.float32, device=ws.device)
    for pol, name in names.items():
        p = kvx.kvx_plan_create(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, cfg.P, cfg.num_groups,
                                kvx.KVX_BF16, cfg.budget[0], cfg.seq_len, cfg.head_group[0], 0,
                                pol)
        kvx.kvx_plan_upload(p)
        w = torch.zeros(p.workspace_bytes() // 4 + 64, dtype=torch.int32, device=ws.device)

        def run():
            kvx.kvx_decode_attn(p, lay.q, lay.k_pools, lay.v_pools, lay.pool_pages, lay.pt,
                                lay.strides, lay.budget, lay.seq_len, 0.0, out, w, stream=stream)
        for _ in range(3):
            run()
        ts = []
        for _ in range(20):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            run()
            b.record(stream)
            b.synchronize()
            ts.append(a.elapsed_time(b) * 1e3)
        st = p.stats()
        tr = torch.zeros((st["num_ctas"], 4), dtype=torch.int64, device=ws.device)
        p.set_trace(tr)
        run()
        torch.cuda.synchronize()
        p.set_trace(None)
        t = tr.cpu().numpy()
        busy = (t[:, 2] - t[:, 1]) / 1e3
        res[name] = {"kernel_us": float(np.median(ts)), "blocks": int(st["num_ctas"]),
                     "block_busy_us_mean": float(busy.mean()), "block_busy_us_max": float(busy.max()),
                     "tokens_per_block_mean": float(st["mean_cta_tokens"]),
                     "tokens_per_block_max": int(st["max_cta_tokens"]),
                     "plan_host_us": float(st["plan_us"])}
        p.destroy()
    return res


def group_sweep(cfg0, table, dev, stream, peak, kvx, torch, layers=4, reps=20):
    """Head-group size G (KV heads sharing one page table) against page
    fragmentation, page-table entries, footprint and kernel throughput, over
    the first `layers` layers (Tangram Figs. 8(c) and 11; G = Hkv is the
    unified page)."""
    from synth.device import TableLayer
    res = {}
    for G in (1, 2, 4, 8):
        if cfg0.Hkv % G:
            continue
        cfg = synth.regroup(cfg0, G)
        plans, lays, alloc, used, entries = [], [], 0, 0, 0
        for l in range(layers):
            p = kvx.kvx_plan_create(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, cfg.P, cfg.num_groups,
                                    kvx.KVX_BF16, cfg.budget[l], cfg.seq_len, cfg.head_group[l], 0)
            kvx.kvx_plan_upload(p)
            st = p.stats()
            alloc += st["slots_allocated"]
            used += st["slots_used"]
            entries += int(p.group_pages().sum())
            plans.append(p)
            lays.append(TableLayer(cfg, l, table, p.group_pages(), seed=0))
        ws = torch.zeros(max(p.workspace_bytes() for p in plans) // 4 + 64, dtype=torch.int32,
                         device=dev)
        out = torch.empty((cfg.B, cfg.Hq, cfg.D), dtype=torch.float32, device=dev)

        def step():
            for l in range(layers):
                L = lays[l]
                kvx.kvx_decode_attn(plans[l], L.q, L.k_pools, L.v_pools, L.pool_pages, L.pt,
                                    L.strides, L.budget, L.seq_len, 0.0, out, ws, stream=stream)
        for _ in range(3):
            step()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            step()
        b.record(stream)
        torch.cuda.synchronize()
        assert kvx.kvx_workspace_status(ws) == 0
        ms = a.elapsed_time(b) / reps
        kvb = sum(cfg.kv_bytes_layer(l) for l in range(layers))
        res[f"G{G}"] = {"groups_per_layer": cfg.num_groups,
                        "fragmentation": 1.0 - used / alloc,
                        "footprint_gb": alloc * 2 * cfg.D * 2 / 1e9,
                        "page_table_entries": entries,
                        "kv_gbs": kvb / (ms * 1e-3) / 1e9,
                        "frac": kvb / (ms * 1e-3) / 1e9 / peak}
        del plans, lays, ws
        torch.cuda.empty_cache()
    return res


def sparse_select(dev, stream, peak, kvx, torch, reps=10):
    """The selection step before sparse decode on one layer of the Llama-3-8B
    shaped workload (batch 8 x 122k, 32/8 heads): score every candidate key
    against the summed GQA query and keep the top 2048 plus the last 128
    (kvx_select_topk), pack the kept rows into pages (kvx_pack_kept), attend
    (kvx_decode_attn); or attend straight over the kept rows of the dense
    cache (kvx_decode_attn_kept). Each stage and both whole pipelines are
    timed. Dense keys and values are tiled from a value table."""
    from synth.device import ValueTable
    cfg = synth.decode_config("llama3_sparse", seed=0, layers=1)
    B, Hq, Hkv, D, L, P = cfg.B, cfg.Hq, cfg.Hkv, cfg.D, int(cfg.seq_len[0]), cfg.P
    top, recent = 2048, 128
    table = ValueTable(seed=31, rows=1 << 18, D=D, dtype="bf16", device=dev)
    keys = torch.empty((B, Hkv, L, D), dtype=torch.bfloat16, device=dev)
    vals = torch.empty_like(keys)
    table.fill(keys, 11)
    table.fill(vals, 77777)
    q = torch.from_numpy(synth.f32_to_bf16_bits(synth.normal(synth.rng(5), (B, Hq, D), "bf16"))
                         .view(np.int16)).view(torch.bfloat16).to(dev)
    sl = torch.from_numpy(cfg.seq_len).to(dev)
    kept = torch.zeros((B * Hkv, top + recent), dtype=torch.int32, device=dev)
    cnt = torch.zeros(B * Hkv, dtype=torch.int32, device=dev)
    sws = torch.zeros(kvx.kvx_select_workspace_bytes(B, Hkv, L) // 4 + 64, dtype=torch.int32,
                      device=dev)
    n = np.full((B, Hkv), top + recent, np.int32)
    hg = np.zeros(Hkv, np.int32)
    plan = kvx.kvx_plan_create(B, Hq, Hkv, D, P, 1, kvx.KVX_BF16, n, cfg.seq_len, hg, 0)
    kvx.kvx_plan_upload(plan)
    gp = plan.group_pages()
    npages = [int(gp.sum())]
    pt = torch.from_numpy(np.arange(npages[0], dtype=np.int32).reshape(B, -1)).to(dev)
    kp = torch.empty((npages[0], Hkv, P, D), dtype=torch.bfloat16, device=dev)
    vp = torch.empty_like(kp)
    aws = torch.zeros(plan.workspace_bytes() // 4 + 64, dtype=torch.int32, device=dev)
    out = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    budget = torch.from_numpy(n.reshape(-1).copy()).to(dev)
    stages = {
        "select": lambda: kvx.kvx_select_topk(keys, q, sl, B, Hq, Hkv, D, L, top, recent, kept,
                                              cnt, sws, stream=stream),
        "pack": lambda: kvx.kvx_pack_kept(plan, keys, vals, L, kept, top + recent, [kp], [vp],
                                          npages, [pt], [pt.shape[1]], aws, stream=stream),
        "attention": lambda: kvx.kvx_decode_attn(plan, q, [kp], [vp], npages, [pt],
                                                 [pt.shape[1]], budget, sl, 0.0, out, aws,
                                                 stream=stream),
        "attention_kept": lambda: kvx.kvx_decode_attn_kept(plan, q, keys, vals, L, kept,
                                                           top + recent, budget, sl, 0.0, out,
                                                           aws, stream=stream),
    }
    # the whole sparse step of one layer, both ways: every call's 2 GB
    # selection pass leaves little of the previous call's rows in L2
    stages["pipeline_packed"] = lambda: (stages["select"](), stages["pack"](),
                                         stages["attention"]())
    stages["pipeline_kept"] = lambda: (stages["select"](), stages["attention_kept"]())
    res = {"workload": f"1 layer, batch {B} x {L} tokens, {Hq} q / {Hkv} KV heads, D {D}, bf16; "
                       f"keep top {top} + last {recent} per head"}
    for name, fn in stages.items():
        for _ in range(3):
            fn()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        res[name] = {"us": a.elapsed_time(b) / reps * 1e3}
    key_bytes = B * Hkv * (L - recent) * D * 2
    res["select"]["keys_gbs"] = key_bytes / (res["select"]["us"] * 1e-6) / 1e9
    res["select"]["frac"] = res["select"]["keys_gbs"] / peak
    kv_kept = B * Hkv * (top + recent) * D * 2 * 2
    res["pack"]["gbs_read_write"] = 2 * kv_kept / (res["pack"]["us"] * 1e-6) / 1e9
    res["attention"]["kv_gbs"] = kv_kept / (res["attention"]["us"] * 1e-6) / 1e9
    res["attention_kept"]["kv_gbs"] = kv_kept / (res["attention_kept"]["us"] * 1e-6) / 1e9
    res["attention"]["note"] = res["attention_kept"]["note"] = (
        "repeated calls over one layer's kept rows (71 MB, which L2 can hold)")
    res["pipeline_packed"]["note"] = "select + pack + attention over the packed pages"
    res["pipeline_kept"]["note"] = "select + attention straight over the kept rows"
    assert kvx.kvx_workspace_status(aws) == 0 and kvx.kvx_workspace_status(sws) == 0
    del keys, vals, kp, vp
    torch.cuda.empty_cache()
    return res


def kvrm_attention(cfg, pools, stagings, bt, dev, stream, peak, steps, kvx, torch):
    """Fixed-shape decode attention after the gather: the K and V staging
    buffers viewed as token-major pages of 16 tokens (identity page table),
    32 query heads over the 8 KV heads, every token kept. Also timed directly
    on the fragmented block pool (block table as page table)."""
    S, mb, Hkv, Hq, D = cfg.S, cfg.max_blocks, 8, 32, 128
    L = np.ascontiguousarray(cfg.seq_tokens, dtype=np.int32)
    plan = kvx.kvx_plan_create(S, Hq, Hkv, D, 16, 1, kvx.KVX_BF16,
                               np.full((S, Hkv), synth.FULL, np.int32), L,
                               np.zeros(Hkv, np.int32), 0, layout=kvx.KVX_LAYOUT_TOKEN_MAJOR)
    kvx.kvx_plan_upload(plan)
    g = synth.rng(77)
    q = torch.from_numpy(synth.f32_to_bf16_bits(synth.normal(g, (S, Hq, D), "bf16")).view(
        np.int16)).view(torch.bfloat16).to(dev)
    out = torch.empty((S, Hq, D), dtype=torch.float32, device=dev)
    ws = torch.zeros(plan.workspace_bytes() // 4 + 64, dtype=torch.int32, device=dev)
    budget = torch.full((S * Hkv,), synth.FULL, dtype=torch.int32, device=dev)
    Ld = torch.from_numpy(L).to(dev)
    ident = torch.arange(S * mb, dtype=torch.int32, device=dev).view(S, mb)
    kv_bytes = int(L.astype(np.int64).sum()) * Hkv * 2 * D * 2
    res = {"workload": f"{S} sequences, {Hq} q / {Hkv} KV heads, D {D}, bf16, all tokens kept"}
    for name, kp, vp, pt, npages in (("over_staging", stagings[0], stagings[1], ident, S * mb),
                                     ("over_fragmented_pool", pools[0], pools[1], bt,
                                      cfg.num_phys)):
        def call():
            kvx.kvx_decode_attn(plan, q, [kp], [vp], [npages], [pt], [pt.shape[1]], budget, Ld,
                                0.0, out, ws, stream=stream)
        for _ in range(3):
            call()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            call()
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / steps
        res[name] = {"value": kv_bytes / (ms * 1e-3) / 1e9, "unit": "GB/s (KV read)",
                     "frac": kv_bytes / (ms * 1e-3) / 1e9 / peak, "ms_per_call": ms}
    assert kvx.kvx_workspace_status(ws) == 0
    return res


def frame_churn(cfg, pools, stagings, dev, stream, peak, kvx, torch, steps, lookahead,
                warm=1500, p_eos=1.0 / 400, p_share=0.25):
    """KV-RM decode loop with runtime variability (KV-RM, Fig. 3): every step
    each live sequence gains a token; a sequence that needs a new block
    Reserves `lookahead` blocks; with probability p_eos a sequence ends (Trim
    to nothing) and a new one takes its slot, sharing a prefix of a random
    live sequence with probability p_share (Alias) before reserving the
    rest; a sequence at the row limit drops its oldest block (Trim). One
    Frame commit per step seals the edits; the coalesced gather then moves
    the committed descriptor's blocks into the staging rows. Times the host
    edits (one batched kvx_frame_edit call per step), the commit (host and
    device) and the gather."""
    import time
    S, M, N = cfg.S, cfg.max_blocks, cfg.num_phys
    bt_tok = 16  # tokens per block of the gather workload
    g = synth.rng(4242 + lookahead)
    f = kvx.Frame(S, M, N)
    tokens = cfg.seq_tokens.astype(np.int64).copy()
    nbv = np.zeros(S, np.int64)

    def need(t):
        return np.minimum(M, -(-t // bt_tok))

    def grow(s, ops):
        want = int(need(tokens[s]))
        if want > nbv[s]:
            c = int(min(M - nbv[s], max(want - nbv[s], lookahead)))
            ops.append((kvx.KVX_EDIT_RESERVE, s, c, 0, 0, 0))
            nbv[s] += c

    def submit(ops):
        if ops:
            st = f.edit(np.asarray(ops, dtype=np.int32))
            assert not st.any(), st

    init = []
    for s in range(S):
        grow(s, init)
    submit(init)

    def edits():
        ops = []
        eos = np.flatnonzero(g.random(S) < p_eos)
        tokens[:] += 1
        for s in eos:
            s = int(s)
            ops.append((kvx.KVX_EDIT_TRIM, s, 0, 0, 0, 0))
            nbv[s] = 0
            tokens[s] = int(g.integers(512, M * bt_tok - 512))
            if g.random() < p_share:
                r = int(g.integers(0, S))
                k = int(min(nbv[r], need(tokens[s]) // 2))
                if r != s and k > 0:
                    ops.append((kvx.KVX_EDIT_ALIAS, s, 0, r, 0, k))
                    nbv[s] = k
        for s in np.flatnonzero(tokens > M * bt_tok):
            s = int(s)
            ops.append((kvx.KVX_EDIT_TRIM, s, 1, int(nbv[s]), 0, 0))
            nbv[s] -= 1
            tokens[s] -= bt_tok
        for s in np.flatnonzero(need(tokens) > nbv):
            grow(int(s), ops)
        submit(ops)

    for _ in range(warm):
        edits()
        f.commit(stream)
    ws = torch.zeros(kvx.kvx_gather_workspace_bytes(S, M) // 4 + 64, dtype=torch.int32,
                     device=dev)

    def gather():
        bt, nb = f.active()
        kvx.kvx_gather_coalesce(bt, nb, S, M, pools, N, cfg.block_bytes, stagings,
                                cfg.row_bytes, 0, ws, stream=stream)

    for _ in range(3):
        edits()
        f.commit(stream)
        gather()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    t_edit = t_commit = 0.0
    records = launches = blocks = 0
    l0, wait0 = f.stats()["launches"], f.stats()["wait_ns"]
    w0 = time.perf_counter()
    for i in range(steps):
        t0 = time.perf_counter()
        edits()
        t1 = time.perf_counter()
        ev[i][0].record(stream)
        f.commit(stream)
        t2 = time.perf_counter()
        ev[i][1].record(stream)
        gather()
        ev[i][2].record(stream)
        t_edit += t1 - t0
        t_commit += t2 - t1
        records += f.stats()["last_records"]
        blocks += int(nbv.sum())
    torch.cuda.synchronize()
    wall_us = (time.perf_counter() - w0) / steps * 1e6
    launches = f.stats()["launches"] - l0
    wait_us = (f.stats()["wait_ns"] - wait0) / 1e3 / steps
    assert kvx.kvx_workspace_status(ws) == 0
    commit_us = sum(e[0].elapsed_time(e[1]) for e in ev) / steps * 1e3
    gather_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / steps
    table, nb, _ = f.state()
    runs = sum(int(1 + np.count_nonzero(np.diff(table[s, :nb[s]]) != 1)) if nb[s] else 0
               for s in range(S))
    moved = 2 * 2 * blocks / steps * cfg.block_bytes  # K and V, read + write
    return {"steps": steps, "lookahead_blocks": lookahead,
            "edit_host_us": t_edit / steps * 1e6,
            "commit_host_us": t_commit / steps * 1e6 - wait_us,
            "commit_wait_us": wait_us,
            "commit_device_us": commit_us, "records_per_step": records / steps,
            "record_bytes_per_step": 8 * records / steps,
            "apply_launches_per_step": launches / steps,
            "gather_ms": gather_ms, "gather_gbs": moved / gather_ms / 1e6,
            "gather_frac": moved / gather_ms / 1e6 / peak,
            "blocks_per_seq": blocks / steps / S, "runs_per_seq": runs / S,
            "step_wall_us": wall_us,
            "submit_share": (t_edit / steps * 1e6 + t_commit / steps * 1e6 - wait_us) / wall_us}


def bench_gather(args, dev, stream, peak, dist, world, rank):
    import torch
    from paged_non_uniform_gb300 import kvx
    from synth.device import ValueTable
    cfg = synth.gather_config(seed=rank_seed(rank))
    table = ValueTable(seed=21 + rank_seed(rank), rows=1 << 18, D=128, dtype="bf16")
    pools, stagings = [], []
    for t in range(2):
        p = torch.empty((cfg.num_phys, cfg.block_bytes // 2), dtype=torch.bfloat16, device=dev)
        table.fill(p, 1000 * t + 7)
        pools.append(p)
        stagings.append(torch.zeros((cfg.S, cfg.row_bytes // 2), dtype=torch.bfloat16,
                                    device=dev))
    bt = torch.from_numpy(cfg.bt).to(dev)
    nb = torch.from_numpy(cfg.nb).to(dev)
    ws = torch.zeros(kvx.kvx_gather_workspace_bytes(cfg.S, cfg.max_blocks) // 4 + 64,
                     dtype=torch.int32, device=dev)

    def call():
        kvx.kvx_gather_coalesce(bt, nb, cfg.S, cfg.max_blocks, pools, cfg.num_phys,
                                cfg.block_bytes, stagings, cfg.row_bytes, 0, ws, stream=stream)

    for _ in range(3):
        call()
    torch.cuda.synchronize()
    steps = max(5, args.steps // 2)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    a.record(stream)
    for _ in range(steps):
        call()
    b.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(a.elapsed_time(b) / steps, dist, dev)
    assert kvx.kvx_workspace_status(ws) == 0
    attn = kvrm_attention(cfg, pools, stagings, bt, dev, stream, peak, steps, kvx, torch)
    frame = None
    if not args.no_frame and rank == 0:
        churn_steps = max(20, min(200, args.steps))
        frame = {"workload": f"{cfg.S} sequences over the same pools: +1 token per step each, "
                             "EOS p=1/400 per sequence and step (Trim), new prompts of 512.."
                             "15872 tokens, 25% sharing half a live prefix (Alias), Reserve "
                             "on demand, oldest block dropped at 16384 tokens (Trim); one "
                             "Frame commit then one coalesced gather per step; 1500 steps of "
                             "churn before timing",
                 "lookahead_1": frame_churn(cfg, pools, stagings, dev, stream, peak, kvx,
                                            torch, churn_steps, 1),
                 "lookahead_8": frame_churn(cfg, pools, stagings, dev, stream, peak, kvx,
                                            torch, churn_steps, 8)}
    live = sum_over_ranks(2 * cfg.live_bytes(), dist, dev)  # K and V, all ranks
    moved = 2 * live                                        # read + write
    return {"workload": f"KV-RM movement: {cfg.S} seqs, {int(cfg.seq_tokens.min())}.."
                        f"{int(cfg.seq_tokens.max())} tokens, 32 KB blocks (16 tok x 8 heads x 128 "
                        f"bf16), K+V pools {2 * cfg.num_phys * cfg.block_bytes / 2**30:.0f} GiB "
                        f"randomly permuted, staging [{cfg.S}][16384] per tensor",
            "value": job_rate(moved, ms), "unit": "GB/s (read+write)",
            "payload_gbs": job_rate(live, ms), "ms_per_call": ms,
            "frac": job_rate(moved, ms) / world / peak, "launches_per_call": 4,
            "attention": attn, "frame_commit": frame}


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world)


if __name__ == "__main__":
    main()
