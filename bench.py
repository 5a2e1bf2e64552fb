#!/usr/bin/env python3
"""Benchmark: one step = indexer score -> top-k select -> sparse attention over
every unit of a workload, through the C ABI of libds4a.so on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--no-cpu-baseline]

Prints one JSON line (rank 0).  Default workload: decode of 32 sequences x 43
layers (1,376 independent caches of 65,536 compressed rows), the decode batch
the HBM roofline is judged on.  Inputs (115 GB) exceed the 126 MB L2 many times
over, so no flush is needed between steps.  With --gpus N (torchrun, one rank
per GPU) every rank runs the whole workload on its own GPU (weak scaling, no
collective on the data path); the timing is the max over ranks.

--impl reference times the fp64 CPU oracle on the host cores on a bounded
sample of the same workload (the slow, obviously-correct statement of the
step), with the same metric and units.
"""
import argparse
import concurrent.futures as cf
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

METRIC = "sparse-attn query-token·layers/s and achieved HBM GB/s (fraction of GB300 peak)"
UNIT = "query-token·layers/s"


def metric_unit(wl):
    """The bench line's metric and unit: the headline's for the attention
    workloads, pooled units per second for the cache-producer workload."""
    if wl.kind == "pool":
        return ("cache-producer units/s (raw push + compressor pooling of the frontier) and achieved HBM GB/s",
                "units/s")
    return METRIC, UNIT
SCALE = 1.0 / math.sqrt(512)


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--workload", default="decode_32x43x65536")
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=15.0, help="CPU work budget of the oracle sample")
    p.add_argument("--units", type=int, default=None,
                   help="decode workloads: run only this many units (small cases for profiling)")
    p.add_argument("--prior-rows", type=int, default=None,
                   help="prefill workload: compressed rows before the chunk (small cases for profiling)")
    p.add_argument("--no-graph", action="store_true",
                   help="launch the C-ABI calls directly in the timed loop instead of replaying a CUDA graph of them")
    p.add_argument("--select", default="auto", choices=["auto", "fused", "two-call"],
                   help="score + top-k: fused (ds4a_indexer_topk) or two calls; auto = fused for decode "
                        "batches of at least one row per SM, two calls otherwise (the faster on each)")
    return p.parse_args()


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), src="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, src="fallback")


# ----------------------------------------------------------------------------
# Clocks during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.lines = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, v in zip(self.NAMES, parts[3:]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def gpu_id_for_smi(torch, dev):
    try:
        u = torch.cuda.get_device_properties(dev).uuid
        return "GPU-" + str(u)
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        return vis.split(",")[dev] if vis else str(dev)


# ----------------------------------------------------------------------------
# Workload arithmetic (algorithmic bytes / flops)
# ----------------------------------------------------------------------------
def decode_bytes(wl):
    """Algorithmic HBM bytes per unit: every indexer key, the selected rows, the
    raw window, q, iq, w, the fp32 output and the selected indices."""
    H = wl.heads
    row_bytes = 512 + 4 if wl.fp8 else 1024           # FP8 store: codes + the row's scale
    per_unit_fixed = wl.top_k * row_bytes + 128 * 1024 + H * 512 * 2 + 64 * 128 * 2 + 64 * 4 + H * 512 * 4 + wl.top_k * 4
    ik = wl.n_rows * 128 * 2
    idx_kernel = wl.n_rows * 256 + 64 * 128 * 2 + 64 * 4
    return wl.units * (ik + per_unit_fixed), wl.units * idx_kernel


def dram_traffic(kernel, units, rows):
    """DRAM bytes (read + write) of one launch of `kernel` on units x rows,
    scaled from the ncu capture recorded in profiles/dram_traffic.json (the
    traffic of these kernels grows in proportion to units x rows).  None when
    there is no capture or the kernel's sources changed since it was taken."""
    import hashlib
    try:
        rec = json.load(open(os.path.join(ROOT, "profiles", "dram_traffic.json")))[kernel]
        m = hashlib.sha256()
        for f in rec["sources"]:
            m.update(open(os.path.join(ROOT, "deepseek_v4_sparse_indexer_gb300", "csrc", f), "rb").read())
        if m.hexdigest() != rec["sources_sha256"]:
            return None
        return rec["dram_bytes"] * (units * rows) / (rec["units"] * rec["rows"])
    except Exception:
        return None


def attn_merge_launches(units, top_k, n_sms):
    """1 when the attention call launches its merge kernel after the attention
    kernel (the library's launch rule: the units left after whole rounds over
    the CTAs are cut into pieces, which the merge kernel combines)."""
    nt = -(-top_k // 64) + 2
    T = units * nt
    G = min(n_sms, 160, T)
    u_rem = units - (units // G) * G
    return 1 if min(u_rem * nt, G) > 1 else 0


def build_fp8_store(pkg, chunks, shape, dev):
    """The FP8 row store (E4M3 codes, power-of-two row scales) of a workload's
    fp32 rows, built chunk by chunk by the library's quantiser (untimed setup)."""
    import torch
    codes = torch.empty(*shape, 512, dtype=torch.uint8, device=dev)
    scale = torch.empty(*shape, dtype=torch.float32, device=dev)
    c2, s2 = codes.view(-1, 512), scale.view(-1)
    for r0, c in chunks:
        pkg.ds4a_rows_to_fp8(c, c2[r0:r0 + c.shape[0]], s2[r0:r0 + c.shape[0]])
    return codes, scale


def pool_bytes(wl, width=512):
    """Algorithmic HBM bytes per launch of the pooling kernel: the fp32 (kv,
    score) frontier and the fp32 pooled row of every unit."""
    return wl.units * (2 * wl.n_rows * width * 4 + width * 4)


def dense_bytes(wl):
    """Algorithmic HBM bytes per unit of a ratio-128 layer: every compressed row,
    the raw window, q, the fp32 output and lse."""
    return wl.units * (wl.n_rows * 1024 + 128 * 1024 + 64 * 512 * 2 + 64 * 512 * 4 + 64 * 4)


def prefill_flops(x, wl):
    import torch
    q_pos = x["q_pos"].cpu().to(torch.int64)
    row_pos = x["row_pos"].cpu().to(torch.int64)
    visible = torch.searchsorted(row_pos, q_pos, right=True)          # rows sorted by position
    idx_flops = float(visible.sum().item()) * 64 * 128 * 2
    # attention: (k selected + window rows) x 64 heads x 512 x 2 (QK) x 2 (PV)
    raw0 = x["raw_pos0"]
    win = torch.clamp(torch.minimum(q_pos - raw0, torch.tensor(x["raw"].shape[0] - 1)) -
                      torch.clamp(q_pos - 127 - raw0, min=0) + 1, min=0)
    rows = torch.clamp(visible, max=wl.top_k) + win
    attn_flops = float(rows.sum().item()) * 64 * 512 * 4
    return idx_flops, attn_flops


# ----------------------------------------------------------------------------
# CPU oracle sample (cpu_baseline leg and the reference arm)
# ----------------------------------------------------------------------------
class OracleSample:
    """A bounded sample of a workload prepared for the fp64 oracle: whole decode
    units (all rows scored, top-k, attention) or prefill queries spread over the
    chunk.  The sample size is calibrated so one timed pass costs about
    `seconds_budget` of CPU work."""

    def __init__(self, wl, seconds_budget, unit_source=None, max_distinct=16):
        import numpy as np
        import torch

        import oracle
        from deepseek_v4_sparse_indexer_gb300.workloads import (make_decode_inputs, make_pool_inputs,
                                                                make_prefill_inputs)

        self.wl = wl
        self.oracle = oracle

        def u16(t):
            return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)

        if wl.kind == "pool":
            x = make_pool_inputs(min(4, wl.units), wl.n_rows, device="cpu", seed=wl.seed)
            pool = [dict(kv=x["kv"][i].numpy(), score=x["score"][i].numpy(), row=x["row"][i].numpy())
                    for i in range(x["kv"].shape[0])]
            t = time.perf_counter()
            self._run(pool[0])
            t1 = time.perf_counter() - t
            n = self._size(seconds_budget, t1, wl.units)
            self.items = [pool[i % len(pool)] for i in range(n)]
            self.text = f"{n} of {wl.units} units (each: raw push of one row + pooling of a {wl.n_rows}-row frontier)"
            return
        if wl.kind in ("decode", "dense"):
            dense = wl.kind == "dense"

            def get_unit(i):
                if unit_source is not None:
                    return unit_source(i)
                x = make_decode_inputs(1, wl.n_rows, device="cpu", seed=wl.seed + 1000 + i,
                                       heavy_frac=wl.heavy_frac, heavy_scale=wl.heavy_scale, with_indexer=not dense,
                                       n_head=wl.heads, with_rows=not wl.fp8)
                if wl.fp8:
                    from deepseek_v4_sparse_indexer_gb300.workloads import decode_rows_fp32_chunks
                    f32 = torch.cat([c for _, c in decode_rows_fp32_chunks(1, wl.n_rows, seed=wl.seed + 1000 + i)])
                    codes, rs = oracle.quantize_rows_fp8(f32.numpy())
                    d = dict(q=u16(x["q"][0]), codes=codes, row_scale=rs, raw=u16(x["raw"][0]), n=wl.n_rows, nraw=128)
                else:
                    d = dict(q=u16(x["q"][0]), rows=u16(x["rows"][0]), raw=u16(x["raw"][0]), n=wl.n_rows, nraw=128)
                if not dense:
                    d.update(iq=u16(x["iq"][0]), w=x["w"][0].numpy(), ik=u16(x["ik"][0]))
                return d

            first = get_unit(0)
            t = time.perf_counter()
            self._run(first)
            t1 = time.perf_counter() - t
            n = self._size(seconds_budget, t1, wl.query_units)
            # At most `pool` distinct units are materialised; the sample cycles
            # through them (the oracle's work per unit does not depend on values).
            pool = [first] + [get_unit(i) for i in range(1, min(n, max_distinct))]
            self.items = [pool[i % len(pool)] for i in range(n)]
            self.text = (f"{n} of {wl.query_units} units (each whole: attention over all {wl.n_rows} rows + "
                         f"128-row window)") if dense else \
                (f"{n} of {wl.query_units} units (each whole: {wl.n_rows} rows scored, top-{wl.top_k}, "
                 f"attention over the selected rows + 128-row window)")
        else:
            x = make_prefill_inputs(wl.queries, wl.extra["prior_rows"], device="cpu", seed=wl.seed,
                                    with_rows=not wl.fp8)
            if wl.fp8:
                from deepseek_v4_sparse_indexer_gb300.workloads import prefill_rows_fp32_chunks
                f32 = torch.cat([c for _, c in prefill_rows_fp32_chunks(x["ik"].shape[0], seed=wl.seed)])
                rows = oracle.quantize_rows_fp8(f32.numpy())
            else:
                rows = u16(x["rows"])
            self.np_in = (u16(x["q"]), u16(x["iq"]), x["w"].numpy(), u16(x["ik"]), rows,
                          x["row_pos"].numpy(), x["q_pos"].numpy(), u16(x["raw"]))
            self.nr = int(x["n_rows"][0])
            self.raw_pos0 = x["raw_pos0"]
            t = time.perf_counter()
            self._run(wl.queries - 1)
            t1 = time.perf_counter() - t
            n = self._size(seconds_budget, t1, wl.queries)
            self.items = [int(v) for v in np.linspace(0, wl.queries - 1, n)]
            self.text = f"{n} of {wl.queries} queries spread over the chunk (first and last included)"

    @staticmethod
    def _size(budget, t1, cap):
        return max(1, min(cap, int(round(budget / max(t1, 1e-3)))))

    def _run(self, item):
        import numpy as np
        wl, o = self.wl, self.oracle
        if wl.kind == "decode" and wl.fp8:
            d = item
            s = o.indexer_score(d["iq"][None], d["w"][None], d["ik"], d["n"])[0]
            idx, _ = o.topk_select(s, wl.top_k)
            o.sparse_attention_fp8(d["q"], d["codes"], d["row_scale"], idx, d["raw"], np.arange(d["nraw"]), SCALE)
        elif wl.kind == "decode":
            d = item
            o.decode_unit(d["q"], d["iq"], d["w"], d["ik"], d["rows"], d["n"], d["raw"], d["nraw"], wl.top_k, SCALE)
        elif wl.kind == "dense":
            d = item
            o.dense_attention(d["q"], d["rows"], d["n"], d["raw"], d["nraw"], SCALE)
        elif wl.kind == "pool":
            d = item
            o.push_raw(np.zeros((128, 512), np.uint16), 128, d["row"])
            o.compressor_pool(d["kv"], d["score"])
        elif wl.fp8:
            q, iq, w, ik, (codes, rs), row_pos, q_pos, raw = self.np_in
            p = int(q_pos[item])
            s = o.indexer_score(iq[item:item + 1], w[item:item + 1], ik, self.nr, q_pos=np.array([p], np.int32),
                                row_pos=row_pos)[0]
            idx, _ = o.topk_select(s, wl.top_k)
            o.sparse_attention_fp8(q[item], codes, rs, idx, raw, o.prefill_window(p, self.raw_pos0, raw.shape[0]), SCALE)
        else:
            q, iq, w, ik, rows, row_pos, q_pos, raw = self.np_in
            o.prefill_query(item, q, iq, w, ik, rows, self.nr, row_pos, q_pos, raw, self.raw_pos0, wl.top_k, SCALE)

    def rate(self, cores):
        """Query-token x layer units per second over the sample, on `cores` threads."""
        t = time.perf_counter()
        with cf.ThreadPoolExecutor(max_workers=cores) as ex:
            list(ex.map(self._run, self.items))
        return len(self.items) / (time.perf_counter() - t)


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# ----------------------------------------------------------------------------
# Reference arm: the oracle on host cores
# ----------------------------------------------------------------------------
# ---------------- multi-process plumbing (one process per GPU, replicas)

def rank_env(environ=None):
    """(rank, world_size, local_rank) as torchrun exports them; one process by default."""
    env = os.environ if environ is None else environ
    return int(env.get("RANK", "0")), int(env.get("WORLD_SIZE", "1")), int(env.get("LOCAL_RANK", "0"))


def rank_seed(base_seed, rank):
    """Each rank's replica of the workload draws its own inputs."""
    return base_seed + rank


def max_over_ranks(values, world, device):
    """Element-wise max over the ranks (all-reduce MAX) of a list of floats:
    the job takes as long as its slowest rank.  The identity in one process."""
    if world == 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t]


def job_value(units_per_rank, world, ms):
    """Whole-job throughput: every rank processes its own units (weak scaling)."""
    return world * units_per_rank / (ms / 1e3)


def run_reference(args, wl):
    rank, _, _ = rank_env()
    if rank != 0:
        return 0
    metric, unit = metric_unit(wl)
    cores = host_cores()
    # Size the sample so that warmup + steps stay within a few minutes of wall time.
    wall_per_step = max(1.0, min(6.0, 90.0 / max(1, args.steps + args.warmup)))
    sample = OracleSample(wl, wall_per_step * cores)
    vals = []
    for i in range(args.warmup + args.steps):
        v = sample.rate(cores)
        if i >= args.warmup:
            vals.append(v)
    value = statistics.median(vals)
    sample_text = sample.text + f", threads={cores}, each step one pass over the sample"
    # A step of this arm is one timed pass over the sample (its units, not the
    # whole workload's): ms_per_step x steps is the time these steps took.
    units_per_step = len(sample.items)
    line = {"impl": "reference", "metric": metric, "value": value, "unit": unit, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": units_per_step / value * 1e3,
            "units_per_step": units_per_step,
            "ms_per_full_workload_extrapolated": wl.query_units / value * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic, seeded (CPU-generated with the same recipe)",
            "config": {"workload": wl.name, "units": wl.units, "queries_per_unit": wl.queries,
                       "rows_per_unit": wl.n_rows, "top_k": wl.top_k, "sampled_units_per_step": units_per_step},
            "cpu_baseline": {"value": value, "unit": unit, "cores": cores, "kind": "oracle", "sample": sample_text},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------
# Our arm
# ----------------------------------------------------------------------------
def main():
    args = parse()
    from deepseek_v4_sparse_indexer_gb300.workloads import WORKLOADS
    if args.workload not in WORKLOADS:
        raise SystemExit(f"unknown workload {args.workload}; choose from {sorted(WORKLOADS)}")
    wl = WORKLOADS[args.workload]
    import dataclasses
    if args.units is not None and wl.kind in ("decode", "dense", "pool"):
        wl = dataclasses.replace(wl, name=f"{wl.name}[units={args.units}]", units=args.units)
    if args.prior_rows is not None and wl.kind == "prefill":
        wl = dataclasses.replace(wl, name=f"{wl.name}[prior_rows={args.prior_rows}]",
                                 n_rows=args.prior_rows + wl.queries // 4, extra=dict(prior_rows=args.prior_rows))
    if args.impl == "reference":
        return run_reference(args, wl)
    metric, unit = metric_unit(wl)
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    import torch
    import torch.distributed as dist

    import deepseek_v4_sparse_indexer_gb300 as pkg
    from deepseek_v4_sparse_indexer_gb300.workloads import (decode_rows_fp32_chunks, make_decode_inputs,
                                                            make_pool_inputs, make_prefill_inputs,
                                                            prefill_rows_fp32_chunks)

    rank, world, local = rank_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    pkg.load()
    pk = peaks()

    def barrier():
        if world > 1:
            dist.barrier()

    seed = rank_seed(wl.seed, rank)
    # auto: the fused select where its candidate kernel (one CTA per row) fills
    # the GPU (decode with as many rows as SMs), or where every row is a
    # candidate anyway (rows of at most 4,096 entries, which the candidate
    # kernel caches whole: 1 x 1,024 rows 27.8 vs 28.4 us per step, ten steps
    # to a graph); the two kernels otherwise (8 x 16,384: 36 vs 89 us;
    # 4 x 262,144: 73 vs 342 us: a few long rows leave the scan's per-CTA
    # thresholds loose, so most rows become candidates).
    n_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    fused = args.select == "fused" or (args.select == "auto" and wl.kind == "decode" and
                                       (wl.units * wl.queries >= n_sms or wl.n_rows <= 4096))
    if wl.kind == "decode":
        x = make_decode_inputs(wl.units, wl.n_rows, device=dev, seed=seed, heavy_frac=wl.heavy_frac,
                               heavy_scale=wl.heavy_scale, n_head=wl.heads, with_rows=not wl.fp8)
        if wl.fp8:
            x["rows8"], x["row_scale"] = build_fp8_store(pkg, decode_rows_fp32_chunks(wl.units, wl.n_rows, dev, seed),
                                                         (wl.units, wl.n_rows), dev)
        new_step = lambda: pkg.DecodeStep(wl.units, wl.n_rows, wl.top_k, device=dev, n_head=wl.heads, fp8=wl.fp8,
                                          fused=fused)
    elif wl.kind == "dense":
        x = make_decode_inputs(wl.units, wl.n_rows, device=dev, seed=seed, with_indexer=False)
        new_step = lambda: pkg.DenseStep(wl.units, wl.n_rows, device=dev)
    elif wl.kind == "pool":
        x = make_pool_inputs(wl.units, wl.n_rows, device=dev, seed=seed)
        new_step = lambda: pkg.ProducerStep(wl.units, device=dev)
    else:
        x = make_prefill_inputs(wl.queries, wl.extra["prior_rows"], device=dev, seed=seed, with_rows=not wl.fp8)
        if wl.fp8:
            n_cap = x["ik"].shape[0]
            x["rows8"], x["row_scale"] = build_fp8_store(pkg, prefill_rows_fp32_chunks(n_cap, dev, seed), (n_cap,), dev)
        new_step = lambda: pkg.PrefillStep(wl.queries, x["ik"].shape[0], wl.top_k, device=dev, fp8=wl.fp8,
                                           fused=fused)
    step = new_step()
    torch.cuda.synchronize()

    for _ in range(args.warmup):
        step(x) if wl.kind == "pool" else step(x, SCALE)
    torch.cuda.synchronize()
    st, flags = pkg.ds4a_get_device_status()
    if st != 0:
        raise SystemExit(f"device status flags {flags} after warm-up")

    # The step's C-ABI calls captured as CUDA graphs, so that host launch gaps
    # do not reach the device time: the whole step as one graph (the timed
    # steps), and the same calls as two graphs (the dominant kernel's part,
    # then the rest) for a second pass over the same steps in which events
    # between the two replays time the dominant part.
    if wl.kind == "dense":
        parts = (lambda: step.attend(x, SCALE), None)
    elif wl.kind == "pool":
        parts = (lambda: step.pool(x), lambda: step.push(x))
    else:
        parts = (lambda: step.score(x), lambda: (step.select(x), step.attend(x, SCALE)))
    whole = lambda: [fn() for fn in parts if fn is not None]
    if not args.no_graph:
        cap = torch.cuda.Stream()
        cap.wait_stream(torch.cuda.current_stream())
        graphs = []
        with torch.cuda.stream(cap):
            for fn in parts + (whole,):
                if fn is None:
                    graphs.append(None)
                    continue
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=cap):
                    fn()
                graphs.append(g)
        torch.cuda.current_stream().wait_stream(cap)
        torch.cuda.synchronize()
        parts = tuple(g.replay if g is not None else None for g in graphs[:2])
        whole = graphs[2].replay
        for _ in range(args.warmup):
            whole()
            parts[0]()
            if parts[1] is not None:
                parts[1]()
        torch.cuda.synchronize()
        st, flags = pkg.ds4a_get_device_status()
        if st != 0:
            raise SystemExit(f"device status flags {flags} after the graph warm-up")

    # ---------------- device-timed region
    K = args.steps
    ev = lambda: torch.cuda.Event(enable_timing=True)
    t0, t1 = ev(), ev()
    sc_s, sc_e = [ev() for _ in range(K)], [ev() for _ in range(K)]
    sampler = ClockSampler(gpu_id_for_smi(torch, dev.index))
    barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    t0.record()
    for i in range(K):
        whole()                                # one step
    t1.record()
    for i in range(K):
        sc_s[i].record()
        parts[0]()                             # the dominant kernel's part: score (+ select when fused),
        sc_e[i].record()                       # the pooling, or the dense attention
        if parts[1] is not None:
            parts[1]()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    barrier()
    ms = t0.elapsed_time(t1) / K
    idx_ms = statistics.mean(a.elapsed_time(b) for a, b in zip(sc_s, sc_e))
    ms, idx_ms = max_over_ranks([ms, idx_ms], world, dev)
    units = wl.query_units
    value = job_value(units, world, ms)

    # ---------------- end to end through the public API with host buffers
    # Every step copies its inputs from pinned host memory and its results back.
    # Two steps are in flight, as in a serving loop: the H2D copy of step i+1's
    # inputs and the D2H copy of step i-1's results run on their own streams
    # (copy engines) while step i's kernels run; events order each buffer's
    # reuse two steps later.
    in_keys = {"dense": ("q",), "pool": ("row", "kv", "score")}.get(wl.kind, ("q", "iq", "w"))
    steps = [step, new_step()]
    xs = [x, dict(x)]
    for k in in_keys:
        xs[1][k] = torch.empty_like(x[k])
    host_in = {k: x[k].cpu().pin_memory() for k in in_keys}
    has_lse = hasattr(step, "lse")
    host_out = [torch.empty(step.out.shape, dtype=step.out.dtype).pin_memory() for _ in range(2)]
    host_lse = [torch.empty(step.lse.shape, dtype=step.lse.dtype).pin_memory() for _ in range(2)] if has_lse else None
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = host_out[0].numel() * 4 + (host_lse[0].numel() * 4 if has_lse else 0)
    for k in in_keys:
        xs[1][k].copy_(x[k])
    steps[1](xs[1]) if wl.kind == "pool" else steps[1](xs[1], SCALE)      # untimed first call of the second step
    torch.cuda.synchronize()
    comp = torch.cuda.current_stream(dev)
    s_h2d, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in, ev_done, ev_out = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    barrier()
    e0, e1 = ev(), ev()
    e0.record(comp)
    s_h2d.wait_stream(comp)
    s_d2h.wait_stream(comp)
    for i in range(K):
        b = i & 1
        if i >= 2:
            s_h2d.wait_event(ev_done[b])        # step i-2 has finished reading these inputs
        with torch.cuda.stream(s_h2d):
            for k, t in host_in.items():
                xs[b][k].copy_(t, non_blocking=True)
        ev_in[b].record(s_h2d)
        comp.wait_event(ev_in[b])
        if i >= 2:
            comp.wait_event(ev_out[b])          # step i-2's results are out of these buffers
        steps[b](xs[b]) if wl.kind == "pool" else steps[b](xs[b], SCALE)
        ev_done[b].record(comp)
        s_d2h.wait_event(ev_done[b])
        with torch.cuda.stream(s_d2h):
            host_out[b].copy_(steps[b].out, non_blocking=True)
            if has_lse:
                host_lse[b].copy_(steps[b].lse, non_blocking=True)
        ev_out[b].record(s_d2h)
    comp.wait_stream(s_d2h)
    comp.wait_stream(s_h2d)
    e1.record(comp)
    torch.cuda.synchronize()
    last = (K - 1) & 1
    if not torch.equal(host_out[last].to(dev), steps[last].out):
        raise SystemExit("end-to-end check: the copied-out result differs from the device result")
    e2e_ms = e0.elapsed_time(e1) / K
    e2e_ms, = max_over_ranks([e2e_ms], world, dev)
    e2e_value = job_value(units, world, e2e_ms)
    st, flags = pkg.ds4a_get_device_status()
    if st != 0:
        raise SystemExit(f"device status flags {flags} after the timed region")

    # ---------------- roofline of the dominant kernel (indexer score; the attention for dense)
    if wl.kind == "pool":
        launches_per_step = 2
    elif wl.kind == "dense":
        launches_per_step = 1 + attn_merge_launches(wl.units, wl.n_rows, n_sms)
    else:
        sub_units = (wl.units if wl.kind == "decode" else wl.queries) * (2 if wl.heads == 128 else 1)
        launches_per_step = 1 + 1 + 1 + attn_merge_launches(sub_units, wl.top_k, n_sms)
        if wl.units * wl.queries <= 76 and not fused and wl.n_rows > (1 << 19):
            launches_per_step += 1            # top-k over few very long rows: a filter pass before the final one
        if fused:
            launches_per_step += 1            # the fused select's counters are zeroed by a kernel of its own
    cfg = {"workload": wl.name, "units": wl.units, "queries_per_unit": wl.queries, "rows_per_unit": wl.n_rows,
           "top_k": wl.top_k if wl.kind != "dense" else "all rows", "raw_window": 128, "heads": wl.heads,
           "head_dim": 512, "indexer": "64x128" if wl.kind != "dense" else "none (ratio-128 layer)",
           "l2": "inputs exceed the L2 many times over; no flush", "parallelism": f"replicas x{world}",
           "peak_source": pk["src"], "rows_store": "fp8 (E4M3 codes + power-of-two row scale)" if wl.fp8 else "bf16",
           "select": ("fused: ds4a_indexer_topk (no scores array)" if fused else
                      "two calls: ds4a_indexer_score then ds4a_topk_select") if wl.kind in ("decode", "prefill")
           else None}
    if wl.kind == "pool":
        pb = pool_bytes(wl)
        achieved = pb / (idx_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm"], "unit": "GB/s",
                "frac": achieved / pk["hbm"], "traffic": None, "kernel": "compressor_pool_kernel",
                "algorithmic_bytes_per_launch": pb, "launch_ms": idx_ms}
        step_bytes = pb + wl.units * (512 * 4 + 512 * 2 + 8)
        cfg.update({"top_k": None, "rows_per_unit": None, "frontier_rows": wl.n_rows, "width": 512,
                    "indexer": None, "heads": None, "head_dim": None})
        cfg["step_algorithmic_bytes"] = step_bytes
        cfg["step_hbm_GBps"] = step_bytes / (ms / 1e3) / 1e9
        cfg["step_hbm_frac"] = cfg["step_hbm_GBps"] / pk["hbm"]
    elif wl.kind == "dense":
        step_bytes = dense_bytes(wl)
        achieved = step_bytes / (idx_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm"], "unit": "GB/s",
                "frac": achieved / pk["hbm"], "traffic": dram_traffic("sparse_attn_kernel", wl.units, wl.n_rows), "kernel": "sparse_attn_kernel",
                "algorithmic_bytes_per_launch": step_bytes, "launch_ms": idx_ms}
        cfg["step_algorithmic_bytes"] = step_bytes
        cfg["step_hbm_GBps"] = step_bytes / (ms / 1e3) / 1e9
        cfg["step_hbm_frac"] = cfg["step_hbm_GBps"] / pk["hbm"]
    elif wl.kind == "decode":
        step_bytes, idx_bytes = decode_bytes(wl)
        achieved = idx_bytes / (idx_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm"], "unit": "GB/s",
                "frac": achieved / pk["hbm"],
                "traffic": dram_traffic("indexer_score_kernel<1>" + ("+fused" if fused else ""), wl.units, wl.n_rows),
                "kernel": "indexer_score_kernel<1>" + (" (fused select) + topk_cand_kernel" if fused else ""),
                "algorithmic_bytes_per_launch": idx_bytes, "launch_ms": idx_ms}
        cfg["step_algorithmic_bytes"] = step_bytes
        cfg["step_hbm_GBps"] = step_bytes / (ms / 1e3) / 1e9
        cfg["step_hbm_frac"] = cfg["step_hbm_GBps"] / pk["hbm"]
    else:
        idx_flops, attn_flops = prefill_flops(x, wl)
        achieved = idx_flops / (idx_ms / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": pk["bf16"], "unit": "TFLOP/s",
                "frac": achieved / pk["bf16"],
                "traffic": dram_traffic("indexer_score_kernel<4>" + ("+fused" if fused else ""), wl.queries, wl.n_rows),
                "kernel": "indexer_score_kernel<4>" + (" (fused select) + topk_cand_kernel" if fused else ""),
                "algorithmic_flops_per_launch": idx_flops, "launch_ms": idx_ms}
        cfg["step_algorithmic_flops"] = idx_flops + attn_flops
        cfg["step_TFLOPs"] = (idx_flops + attn_flops) / (ms / 1e3) / 1e12
        cfg["step_tensor_frac"] = cfg["step_TFLOPs"] / pk["bf16"]

    line = {"metric": metric, "value": value, "unit": unit, "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": ("synthetic: seeded fp32 frontiers, kv N(0,1)/sqrt(512), scores N(0,1)" if wl.kind == "pool" else
                     "synthetic: seeded N(0,1)/sqrt(d) bf16 rows/keys/queries, fp16 raw window, U(0,1) weights"),
            "config": cfg, "roofline": roof,
            "e2e": {"value": e2e_value, "unit": unit, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": e2e_ms,
                    "note": (("per step: H2D of the new rows and the (kv, score) frontiers from pinned memory, the "
                             "push and pooling C-ABI ops, D2H of the pooled rows") if wl.kind == "pool" else
                            ("per step: H2D of q from pinned memory, the dense attention C-ABI op, D2H of out and "
                             "lse; the KV caches stay resident in HBM") if wl.kind == "dense" else
                            ("per step: H2D of the queries (q, iq, w) from pinned memory, the three C-ABI ops, D2H "
                             "of out and lse; the KV caches stay resident in HBM")) +
                            "; two steps in flight: the copies of steps i+1 and i-1 overlap step i's kernels"},
            "gpu_launches": launches_per_step * K, "clocks": clocks,
            "launch": "CUDA graph replay of the step's C-ABI calls" if not args.no_graph else "direct C-ABI calls"}

    # ---------------- CPU baseline: the oracle on the host cores (rank 0, N = 1)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import numpy as np
        cores = host_cores()

        def u16(t):
            return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)

        unit_source = None
        if wl.kind == "decode" and not wl.fp8:
            def unit_source(i):
                u = (i * 7919) % wl.units
                return dict(q=u16(x["q"][u]), iq=u16(x["iq"][u]), w=x["w"][u].cpu().numpy(), ik=u16(x["ik"][u]),
                            rows=u16(x["rows"][u]), raw=u16(x["raw"][u]), n=wl.n_rows, nraw=128)
        elif wl.kind == "pool":
            unit_source = None
        elif wl.kind == "dense":
            def unit_source(i):
                u = (i * 7919) % wl.units
                return dict(q=u16(x["q"][u]), rows=u16(x["rows"][u]), raw=u16(x["raw"][u]), n=wl.n_rows, nraw=128)
        sample = OracleSample(wl, args.cpu_seconds, unit_source)
        v = sample.rate(cores)
        line["cpu_baseline"] = {"value": v, "unit": unit, "cores": cores, "kind": "oracle",
                                "sample": sample.text + f", threads={cores}"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
