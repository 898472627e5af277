#!/usr/bin/env python3
"""Benchmark of the hd512 attention hot path on GB300.

One step = one pass of the whole path on synthetic inputs already resident in
HBM: the chunked causal prefill (8192 query rows at positions 8192..16383
against 16384 keys, 32 query heads over 4 KV heads, head dim 512) plus the
paged split-K decode over the nine decode shapes (batch {1,16,64} x KV length
{4096,16384,28672}, 8 query heads over 4 KV heads, page size 64).  L2 is
flushed (a 512 MiB write) before every step; kernels are timed with CUDA
events on the launching stream.

Headline `value`: prefill TFLOP/s = 4 * 512 * n_q_heads * (visible query-key
pairs) / prefill time (the FLOP convention that reproduces the 131 TFLOP the
RTX PRO 6000 page states for 10 global layers of a 19,985-token prompt).
Decode is reported as HBM GB/s of live K/V bytes.

Further legs, each timed on its own with L2 flushed before every call (keys
of the JSON line): `e2e` (the prefill with its inputs copied in from pinned
host memory and its outputs copied back every step), `prefill_paged` (the
chunked config and a mixed batch through a paged cache), `local256` (head dim
256 under a 1,024-key window), `decode_fp8` (the nine decode shapes over an
FP8 E4M3 cache), `decode_q` (4 query tokens per sequence, batch 64 x kv
16384), `prefill_full`, `prefill_full_stress` (20480 x 20480 causal, 32/4
heads; the stress variant multiplies every 64th key row by 8) and
`prefill_mqa` (49152 x 49152 causal, 16 query heads over 1 KV head), each
with its own `roofline`; `cpu_baseline` (the fp64 oracle on a bounded row
sample of the chunked config, and under `plan` the oracle in full on the
tiny and batch-1 decode configs and per-row on stratified samples of the
large configs, with a labelled extrapolation).  The
`roofline` objects carry DRAM traffic per launch from `profiles/
dram_traffic.txt` when it was captured on the current source.

`--impl reference` times the fp64 CPU oracle on a bounded row sample of the
same workload (the reference arm of this benchmark).
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

HEAD_DIM = 512
PREFILL = dict(name="chunked", seqlen_q=8192, seqlen_k=16384, q_offset=8192, n_q_heads=32,
               n_kv_heads=4)
DECODE_SHAPES = [(b, n) for b in (1, 16, 64) for n in (4096, 16384, 28672)]
DECODE_HEADS = (8, 4)
# several query tokens per sequence (the last q_len positions of the cache)
DECODE_Q_SHAPE = {"batch": 64, "kv_len": 16384, "q_len": 4}
PAGE = 64
# prefill over a paged cache: (chunk rows, cached positions incl. the chunk) per sequence.
# "chunked": the headline chunk through shuffled 64-key pages; "varlen": a mixed batch.
# FP8 E4M3 cache: per-tensor scales of the synthetic cache (N(0,1) / scale -> e4m3)
FP8_SCALES = (1 / 32, 1 / 32)
# the sliding-window local layers: heads of 256 dimensions over the last 1,024 tokens
LOCAL256 = {"seqlen": 20480, "window": 1024, "n_q_heads": 32, "n_kv_heads": 4}
# the large prefill configs, each timed as a leg of its own
PREFILL_LEGS = {
    "prefill_full": dict(seqlen_q=20480, seqlen_k=20480, q_offset=0, n_q_heads=32, n_kv_heads=4,
                         stress=False),
    "prefill_full_stress": dict(seqlen_q=20480, seqlen_k=20480, q_offset=0, n_q_heads=32,
                                n_kv_heads=4, stress=True),
    "prefill_mqa": dict(seqlen_q=49152, seqlen_k=49152, q_offset=0, n_q_heads=16, n_kv_heads=1,
                        stress=False),
}
PAGED_PREFILL = {
    "chunked": [(8192, 16384)],
    "varlen": [(8192, 8192), (4096, 12288), (2048, 20480), (1024, 1024), (3000, 7000)],
}
METRIC = "hd512 causal prefill TFLOP/s (% of GB300 BF16 peak); decode HBM GB/s"
PREFILL_WORKLOAD = ("chunked prefill: 8192 q rows at positions 8192..16383 vs 16384 keys, "
                    "32 q / 4 kv heads, d512, causal, bf16 N(0,1)")
DECODE_WORKLOAD = ("; paged decode b{1,16,64} x kv{4096,16384,28672}, 8/4 heads, page 64, "
                   "num_splits auto")


def visible_pairs(seqlen_q: int, seqlen_k: int, q_offset: int, causal: bool = True,
                  window: int = 0) -> int:
    """Number of (query row, key) pairs the mask lets through, per query head."""
    total = 0
    # closed form per row is cheap enough in Python for these sizes
    for i in range(seqlen_q):
        p = q_offset + i
        hi = min(seqlen_k, p + 1) if causal else seqlen_k
        lo = max(0, p - window + 1) if window > 0 else 0
        if hi > lo:
            total += hi - lo
    return total


def prefill_flops(seqlen_q, seqlen_k, q_offset, n_q_heads, causal=True, window=0,
                  head_dim=HEAD_DIM) -> int:
    return 4 * head_dim * n_q_heads * visible_pairs(seqlen_q, seqlen_k, q_offset, causal, window)


def decode_bytes(batch: int, kv_len: int, n_q_heads: int, n_kv_heads: int, q_len: int = 1,
                 kv_elem_bytes: int = 2) -> int:
    """Algorithmic HBM bytes of one decode call: live K and V rows (2 bytes an
    element in bf16, 1 in FP8 E4M3), q, out, lse, page table and lengths (the
    split partials are not counted)."""
    kv = batch * kv_len * n_kv_heads * HEAD_DIM * kv_elem_bytes * 2
    qo = q_len * (batch * n_q_heads * HEAD_DIM * 2 * 2 + batch * n_q_heads * 4)
    pt = batch * ((kv_len + PAGE - 1) // PAGE) * 4 + batch * 4
    return kv + qo + pt


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def source_digest(names) -> str:
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "head_dim_flashattention_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def max_over_ranks(values, device):
    """Each timing taken as the slowest rank's (an all-reduce MAX over the
    process group when one is initialised with more than one rank)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return list(values)
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_rate(units_per_step_per_rank: float, steps: int, world: int, seconds: float) -> float:
    """Whole-job throughput: the units every rank processed over the slowest rank's time."""
    return units_per_step_per_rank * steps * world / seconds


def recorded_traffic(kernel: str, digest: str):
    """DRAM bytes per launch recorded from an ncu capture of this exact kernel
    source, or None when absent or taken on older source."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    try:
        with open(path) as f:
            for line in f:
                if line.startswith("#") or not line.strip():
                    continue
                kv = dict(tok.split("=", 1) for tok in line.split())
                if kv.get("kernel") == kernel and kv.get("src") == digest:
                    return float(kv["bytes_per_launch"])
    except (OSError, ValueError, KeyError):
        return None
    return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.tmp = None

    def start(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.tmp, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.tmp.flush()
        self.tmp.seek(0)
        sms, maxes, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.tmp.read().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1]))
                maxes.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.tmp.name)
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        hi = max(sms)
        loaded = [s for s in sms if s >= 0.5 * hi] or sms
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(maxes),
                "reasons": sorted(reasons), "samples": len(sms),
                "power_w_max": max(power) if power else None}


def leg_sampler(device):
    """A started ClockSampler for one separately timed leg (its calls run back
    to back, so its clocks and power reasons can differ from the main step's)."""
    cs = ClockSampler(device.index if device.index is not None else 0)
    cs.start()
    time.sleep(0.2)
    return cs


# ------------------------------------------------------------------ CPU oracle

_ORACLE_INPUTS = {}


def _stratified_rows(seqlen_q: int, q_offset: int, tokens_per_tile: int, stress: bool,
                     budget: int) -> list:
    """A bounded stratified row sample: the first and last rows, rows on both
    sides of q-tile boundaries near the start, middle and end, the rows just
    after two stressed keys (stress variant), and evenly spaced rows up to
    `budget` rows in all."""
    n = seqlen_q
    rows = {0, 1, n - 2, n - 1}
    for t in (tokens_per_tile, (n // (2 * tokens_per_tile)) * tokens_per_tile,
              (n // tokens_per_tile - 1) * tokens_per_tile):
        rows.update(x for x in (t - 1, t) if 0 <= x < n)
    if stress:
        for j in (64 * 3, 64 * (n // 128)):
            i = j - q_offset
            rows.update(x for x in (i, i + 1) if 0 <= x < n)
    spare = max(0, budget - len(rows))
    if spare:
        rows.update(int(x) for x in np.linspace(0, n - 1, spare + 2)[1:-1])
    return sorted(rows)


def oracle_sample(budget_rows: int = 24, decode_batch: int = 1, decode_len: int = 4096):
    """Times the fp64 oracle on a bounded sample of the chunked prefill
    workload.  Returns (flops, seconds, threads, description)."""
    import oracle
    from head_dim_flashattention_gb300 import workloads

    cfg = workloads.PREFILL_CONFIGS["chunked"]
    if "chunked" not in _ORACLE_INPUTS:
        _ORACLE_INPUTS["chunked"] = workloads.prefill_inputs(cfg)
    q, k, v = _ORACLE_INPUTS["chunked"]
    rows = [int(x) for x in np.linspace(0, cfg.seqlen_q - 1, budget_rows)]
    threads = oracle.default_threads()
    t0 = time.perf_counter()
    oracle.prefill(q, k, v, q_offset=cfg.q_offset, scale=cfg.scale, rows=rows, threads=threads)
    dt = time.perf_counter() - t0
    flops = sum(4 * HEAD_DIM * cfg.n_q_heads * min(cfg.seqlen_k, cfg.q_offset + r + 1)
                for r in rows)
    desc = ("oracle_prefill on %d evenly spaced query rows (all 32 heads) of the chunked "
            "config: %.3g GFLOP" % (len(rows), flops / 1e9))
    return flops, dt, threads, desc


def oracle_plan(rows_per_config: int = 16):
    """The fp64 oracle on the host cores, as the CPU baseline plan asks:
    in full on the tiny prefill config and on the batch-1 decode configs;
    on a stratified row sample of the chunked, full (and stress) and MQA
    prefill configs, as seconds per row and a labelled extrapolation to the
    whole config (the cost of a row grows with its visible keys)."""
    import torch

    import oracle
    from head_dim_flashattention_gb300 import workloads

    threads = oracle.default_threads()
    res = {"cores": threads, "kind": "oracle"}
    # tiny prefill in full
    cfg = workloads.PREFILL_CONFIGS["tiny"]
    q, k, v = workloads.prefill_inputs(cfg)
    t0 = time.perf_counter()
    oracle.prefill(q, k, v, q_offset=cfg.q_offset, scale=cfg.scale, causal=cfg.causal,
                   threads=threads)
    dt = time.perf_counter() - t0
    fl = prefill_flops(cfg.seqlen_q, cfg.seqlen_k, cfg.q_offset, cfg.n_q_heads)
    res["tiny_full"] = {"seconds": dt, "TFLOP/s": fl / dt / 1e12, "flops": fl,
                        "what": "tiny prefill 256x256, 8/1 heads, every row (full config)"}
    # batch-1 decode configs in full (GB/s of live K/V, as the GPU leg)
    dec = {}
    for n in (4096, 16384, 28672):
        dc = workloads.DECODE_CONFIGS["b1_kv%d" % n]
        pc = workloads.decode_inputs(dc)
        t0 = time.perf_counter()
        oracle.decode_paged(pc.q, pc.k_pages, pc.v_pages, pc.page_table, pc.kv_lens,
                            threads=threads)
        dt = time.perf_counter() - t0
        by = decode_bytes(1, n, dc.n_q_heads, dc.n_kv_heads)
        dec["b1_kv%d" % n] = {"seconds": dt, "GB/s": by / dt / 1e9, "bytes": by}
    res["decode_full"] = dec
    # large prefill configs: stratified rows, seconds per row, extrapolation
    big = {}
    for name, cname in (("chunked", "chunked"), ("full", "full"), ("full_stress", "full_stress"),
                        ("mqa", "mqa")):
        c = workloads.PREFILL_CONFIGS[cname]
        g = c.n_q_heads // c.n_kv_heads
        rows = _stratified_rows(c.seqlen_q, c.q_offset, 128 // g, c.stress, rows_per_config)
        # Q only for the sampled rows (the same distribution); every key
        qs = workloads.randn_bf16((len(rows), c.n_q_heads, HEAD_DIM), c.seed * 3 + 7)
        key = ("kv", c.seqlen_k, c.n_kv_heads, c.stress)
        if key not in _ORACLE_INPUTS:
            kk = workloads.randn_bf16((c.seqlen_k, c.n_kv_heads, HEAD_DIM), c.seed * 3 + 1)
            vv = workloads.randn_bf16((c.seqlen_k, c.n_kv_heads, HEAD_DIM), c.seed * 3 + 2)
            if c.stress:
                kk[::64] *= 8
            _ORACLE_INPUTS[key] = (kk, vv)
        kk, vv = _ORACLE_INPUTS[key]
        t0 = time.perf_counter()
        for i, r in enumerate(rows):
            oracle.prefill(qs[i:i + 1], kk, vv, q_offset=c.q_offset + r, scale=c.scale,
                           causal=True, threads=threads)
        dt = time.perf_counter() - t0
        fl_sample = sum(4 * HEAD_DIM * c.n_q_heads * min(c.seqlen_k, c.q_offset + r + 1)
                        for r in rows)
        fl_all = prefill_flops(c.seqlen_q, c.seqlen_k, c.q_offset, c.n_q_heads)
        big[name] = {"rows": len(rows), "seconds": dt, "seconds_per_row": dt / len(rows),
                     "TFLOP/s": fl_sample / dt / 1e12,
                     "extrapolated_seconds_whole_config": dt * fl_all / fl_sample,
                     "extrapolation": "measured seconds x (config FLOP / sample FLOP); "
                                      "not measured"}
        del qs
    res["prefill_sampled"] = big
    return res


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    # warm-up steps, then K timed steps, each a bounded oracle sample
    for _ in range(args.warmup):
        oracle_sample(budget_rows=2)
    flops_total, secs = 0, 0.0
    threads, desc = 1, ""
    for _ in range(args.steps):
        f, dt, threads, desc = oracle_sample(budget_rows=args.ref_rows)
        flops_total += f
        secs += dt
    value = flops_total / secs / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": PREFILL_WORKLOAD, "l2": "n/a (host CPU)",
                   "parallelism": "host threads"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line))
    return 0


# ------------------------------------------------------------------ GPU arm

def time_decode_fp8(args, fa, g, dev, stream, shapes, flush, world, peaks):
    """The decode shapes (q_len 1, 8/4 heads, page 64, num_splits auto) over an
    FP8 E4M3 cache: every step flushes L2, then calls each shape once."""
    import torch

    hq, hk = DECODE_HEADS
    ks, vs = FP8_SCALES
    gcpu = torch.Generator()
    gcpu.manual_seed(0x5EED + 8)
    legs = []
    for b, n in shapes:
        npg = (n + PAGE - 1) // PAGE
        shape = (b * npg, PAGE, hk, HEAD_DIM)
        kp = (torch.randn(shape, generator=g, device=dev) / ks).to(torch.float8_e4m3fn)
        vp = (torch.randn(shape, generator=g, device=dev) / vs).to(torch.float8_e4m3fn)
        pt = torch.randperm(b * npg, generator=gcpu).to(torch.int32).view(b, npg).to(dev)
        legs.append(dict(b=b, n=n, kp=kp, vp=vp, pt=pt,
                         kl=torch.full((b,), n, dtype=torch.int32, device=dev),
                         q=torch.randn((b, hq, HEAD_DIM), generator=g, device=dev).to(torch.bfloat16),
                         out=torch.empty((b, hq, HEAD_DIM), dtype=torch.bfloat16, device=dev),
                         lse=torch.empty((b, hq), dtype=torch.float32, device=dev),
                         ws=torch.empty(fa.fa512_decode_workspace_bytes_fp8(b, 1, hq, hk, PAGE, n, 0),
                                        dtype=torch.uint8, device=dev),
                         bytes=decode_bytes(b, n, hq, hk, kv_elem_bytes=1)))

    def call(d):
        fa.fa512_decode_paged_fp8(d["q"], d["kp"], d["vp"], d["pt"], d["kl"], d["out"], d["lse"],
                                  k_scale=ks, v_scale=vs, max_kv_len=d["n"], workspace=d["ws"],
                                  stream=stream)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        for d in legs:
            call(d)
    torch.cuda.synchronize()
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in legs] for _ in range(args.steps)]
    cs = leg_sampler(dev)
    for s in range(args.steps):
        flush.zero_()
        for i, d in enumerate(legs):
            evs[s][i][0].record(stream)
            call(d)
            evs[s][i][1].record(stream)
    torch.cuda.synchronize()
    clocks = cs.stop()
    ms = [sum(evs[s][i][0].elapsed_time(evs[s][i][1]) for s in range(args.steps)) / args.steps
          for i in range(len(legs))]
    ms = max_over_ranks(ms, dev)
    total_bytes = sum(d["bytes"] for d in legs)
    gbs = job_rate(total_bytes, args.steps, world, sum(ms) * args.steps / 1e3) / 1e9
    per = {"b%d_kv%d" % (d["b"], d["n"]): {"ms": m, "GB/s": d["bytes"] / m / 1e6,
                                            "splits": fa.fa512_decode_auto_splits_fp8(d["b"], 1, hq, hk, PAGE, d["n"])}
           for d, m in zip(legs, ms)}
    return {"workload": "paged decode b{1,16,64} x kv{4096,16384,28672}, 8/4 heads, page 64, "
                        "num_splits auto, FP8 E4M3 K/V cache (per-tensor scales 1/32)",
            "value": gbs, "unit": "GB/s", "ms": sum(ms), "bytes_per_step": total_bytes,
            "frac_of_measured_hbm": gbs / world / peaks["hbm_gbs"],
            "kernel": "fa512::decode::mma8::decode_fp8_mma_kernel + merge",
            "traffic_b64_kv28672": recorded_traffic(
                "decode_fp8_mma_kernel", source_digest(["decode_sm103.cu", "fa512_device.cuh",
                                                        "fa512_internal.h"])),
            "l2": "flushed before every step (each shape called once per step)",
            "clocks": clocks, "per_shape": per}


def run_ours(args):
    import torch
    import torch.distributed as dist

    import head_dim_flashattention_gb300 as fa
    from head_dim_flashattention_gb300 import build as libbuild

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if rank == 0:
        libbuild.build()
    if world > 1:
        dist.barrier()
    fa.load_library()
    stream = torch.cuda.current_stream()

    # ---- resident inputs (seeded, drawn on the device)
    g = torch.Generator(device=dev)
    g.manual_seed(0x5EED + 2 + 1000 * rank)
    P = PREFILL
    q = torch.randn((P["seqlen_q"], P["n_q_heads"], HEAD_DIM), generator=g, device=dev,
                    dtype=torch.float32).to(torch.bfloat16)
    k = torch.randn((P["seqlen_k"], P["n_kv_heads"], HEAD_DIM), generator=g, device=dev,
                    dtype=torch.float32).to(torch.bfloat16)
    v = torch.randn(k.shape, generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
    out = torch.empty_like(q)
    lse = torch.empty((P["n_q_heads"], P["seqlen_q"]), dtype=torch.float32, device=dev)
    pf_flops = prefill_flops(P["seqlen_q"], P["seqlen_k"], P["q_offset"], P["n_q_heads"])

    hq, hk = DECODE_HEADS
    dec = []
    shapes = DECODE_SHAPES
    if args.decode_shapes:
        want = set(args.decode_shapes.split(","))
        shapes = [(b, n) for b, n in DECODE_SHAPES if "b%d_kv%d" % (b, n) in want]
    if not args.no_decode:
        gcpu = torch.Generator()
        gcpu.manual_seed(0x5EED + 5)
        for b, n in shapes:
            npg = (n + PAGE - 1) // PAGE
            num_pages = b * npg
            kp = torch.randn((num_pages, PAGE, hk, HEAD_DIM), generator=g, device=dev,
                             dtype=torch.float32).to(torch.bfloat16)
            vp = torch.randn((num_pages, PAGE, hk, HEAD_DIM), generator=g, device=dev,
                             dtype=torch.float32).to(torch.bfloat16)
            perm = torch.randperm(num_pages, generator=gcpu).to(torch.int32)
            pt = perm.view(b, npg).to(dev)
            kl = torch.full((b,), n, dtype=torch.int32, device=dev)
            dq = torch.randn((b, hq, HEAD_DIM), generator=g, device=dev,
                             dtype=torch.float32).to(torch.bfloat16)
            ws = torch.empty(fa.fa512_decode_workspace_bytes(b, hq, hk, PAGE, n, 0),
                             dtype=torch.uint8, device=dev)
            dec.append(dict(b=b, n=n, kp=kp, vp=vp, pt=pt, kl=kl, q=dq, ws=ws,
                            out=torch.empty((b, hq, HEAD_DIM), dtype=torch.bfloat16, device=dev),
                            lse=torch.empty((b, hq), dtype=torch.float32, device=dev),
                            bytes=decode_bytes(b, n, hq, hk),
                            splits=fa.fa512_decode_auto_splits(b, hk, PAGE, n)))
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    torch.cuda.synchronize()

    def step(events):
        flush.zero_()
        events[0].record(stream)
        if not args.no_prefill:
            fa.fa512_prefill(q, k, v, out, lse, q_offset=P["q_offset"], causal=True, stream=stream)
        events[1].record(stream)
        for i, d in enumerate(dec):
            fa.fa512_decode_paged(d["q"], d["kp"], d["vp"], d["pt"], d["kl"], d["out"], d["lse"],
                                  max_kv_len=d["n"], workspace=d["ws"], stream=stream)
            events[2 + i].record(stream)

    n_ev = 2 + len(dec)
    for _ in range(args.warmup):
        step([torch.cuda.Event(enable_timing=True) for _ in range(n_ev)])
    torch.cuda.synchronize()
    assert fa.fa512_device_status() == 0

    sampler = ClockSampler(local)
    all_events = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
                  for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    t_wall = time.perf_counter()
    for s in range(args.steps):
        step(all_events[s])
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_wall
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    status = fa.fa512_device_status()

    pf_ms = [e[0].elapsed_time(e[1]) for e in all_events]
    dec_ms = [[e[1 + i].elapsed_time(e[2 + i]) for i in range(len(dec))] for e in all_events]
    step_ms = [pf_ms[s] + sum(dec_ms[s]) for s in range(args.steps)]
    t_pf = sum(pf_ms) / 1e3
    t_dec = sum(sum(x) for x in dec_ms) / 1e3
    t_step = sum(step_ms) / 1e3
    t_pf, t_dec, t_step, wall = max_over_ranks([t_pf, t_dec, t_step, wall], dev)

    value = job_rate(pf_flops, args.steps, world, t_pf) / 1e12 if not args.no_prefill else None
    dec_bytes = sum(d["bytes"] for d in dec)
    dec_gbs = job_rate(dec_bytes, args.steps, world, t_dec) / 1e9 if dec else None

    peaks, peak_kind = read_peaks()
    pf_avg_s = t_pf / args.steps if not args.no_prefill else float("nan")
    pf_src = source_digest(["prefill_so_sm103.cu", "fa512_pair.cuh", "fa512_device.cuh", "fa512_internal.h"])
    dec_src = source_digest(["decode_sm103.cu", "fa512_device.cuh", "fa512_internal.h"])
    roofline = {"kernel": "fa512::prefill_so::prefill_so_kernel<false>", "bound": "tensor",
                "achieved": pf_flops / pf_avg_s / 1e12, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": pf_flops / pf_avg_s / 1e12 / peaks["bf16_tflops"],
                "peak_kind": "%s burst bf16 (MEASURED_PEAKS.json)" % peak_kind,
                "frac_of_sustained": pf_flops / pf_avg_s / 1e12 / peaks["bf16_tflops_sustained"],
                "frac_of_nominal_2250": pf_flops / pf_avg_s / 1e12 / 2250.0,
                "traffic": recorded_traffic("prefill_so_kernel", pf_src), "src": pf_src}
    decode_roofline = None
    if dec:
        per = {}
        for i, d in enumerate(dec):
            ms = sum(dec_ms[s][i] for s in range(args.steps)) / args.steps
            per["b%d_kv%d" % (d["b"], d["n"])] = {"ms": ms, "GB/s": d["bytes"] / ms / 1e6,
                                                  "splits": d["splits"]}
        decode_roofline = {"kernel": "fa512::decode (split + merge)", "bound": "hbm",
                           "achieved": dec_gbs / world, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                           "frac": dec_gbs / world / peaks["hbm_gbs"],
                           "frac_of_8000": dec_gbs / world / 8000.0,
                           # DRAM bytes of the largest shape's split kernel (b64 x kv28672
                           # runs the tensor-core streaming kernel)
                           "traffic": recorded_traffic("decode_bf16_mma_kernel", dec_src),
                           "traffic_shape": "b64_kv28672",
                           "src": dec_src, "per_shape": per}

    # ---- end to end through the public API with host buffers.  Every step
    # copies its Q/K/V in from pinned host memory and its O/LSE back out; the
    # copies of neighbouring steps overlap the kernel on their own streams
    # (inputs and outputs double-buffered on the device), as a serving loop
    # would run them.
    e2e = None
    if not args.no_e2e and not args.no_prefill:
        qh = q.cpu().pin_memory()
        kh = k.cpu().pin_memory()
        vh = v.cpu().pin_memory()
        dev_in = [(torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)) for _ in range(2)]
        dev_out = [(torch.empty_like(out), torch.empty_like(lse)) for _ in range(2)]
        host_out = [(torch.empty(out.shape, dtype=out.dtype).pin_memory(),
                     torch.empty(lse.shape, dtype=lse.dtype).pin_memory()) for _ in range(2)]
        s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

        def e2e_run(n_steps):
            in_ready = [torch.cuda.Event() for _ in range(2)]
            done = [torch.cuda.Event() for _ in range(2)]
            copied = [torch.cuda.Event() for _ in range(2)]
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0.record(s_in)
            for i in range(n_steps):
                b = i & 1
                qd, kd, vd = dev_in[b]
                od, ld = dev_out[b]
                with torch.cuda.stream(s_in):
                    if i >= 2:
                        s_in.wait_event(done[b])          # step i-2 finished reading dev_in[b]
                    qd.copy_(qh, non_blocking=True)
                    kd.copy_(kh, non_blocking=True)
                    vd.copy_(vh, non_blocking=True)
                    in_ready[b].record(s_in)
                stream.wait_event(in_ready[b])
                if i >= 2:
                    stream.wait_event(copied[b])          # step i-2's result left dev_out[b]
                flush.zero_()
                fa.fa512_prefill(qd, kd, vd, od, ld, q_offset=P["q_offset"], causal=True,
                                 stream=stream)
                done[b].record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(done[b])
                    host_out[b][0].copy_(od, non_blocking=True)
                    host_out[b][1].copy_(ld, non_blocking=True)
                    copied[b].record(s_out)
            s_out.wait_event(done[(n_steps - 1) & 1])
            t1.record(s_out)
            torch.cuda.synchronize()
            return t0.elapsed_time(t1) / 1e3

        e2e_run(3)
        (t_e2e,) = max_over_ranks([e2e_run(args.steps)], dev)
        h2d = (q.numel() + k.numel() + v.numel()) * 2
        d2h = out.numel() * 2 + lse.numel() * 4
        e2e = {"value": job_rate(pf_flops, args.steps, world, t_e2e) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "what": "fa512_prefill with pinned-host Q/K/V copied in and O/LSE copied out "
                       "every step, copies of neighbouring steps overlapping the kernel on two "
                       "more streams (L2 flush included)"}

    # ---- prefill over a paged cache (varlen batches), timed on its own
    prefill_paged = None
    if not args.no_prefill and not args.no_paged:
        prefill_paged = {}
        gcpu = torch.Generator()
        gcpu.manual_seed(0x5EED + 7)
        hq_p, hk_p = P["n_q_heads"], P["n_kv_heads"]
        for name, seqs in PAGED_PREFILL.items():
            npgs = [(n + PAGE - 1) // PAGE for _, n in seqs]
            num_pages = sum(npgs)
            kp = torch.randn((num_pages, PAGE, hk_p, HEAD_DIM), generator=g, device=dev,
                             dtype=torch.float32).to(torch.bfloat16)
            vp = torch.randn(kp.shape, generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
            perm = torch.randperm(num_pages, generator=gcpu).to(torch.int32)
            pt = torch.zeros((len(seqs), max(npgs)), dtype=torch.int32)
            c = 0
            for i, m in enumerate(npgs):
                pt[i, :m] = perm[c:c + m]
                c += m
            pt = pt.to(dev)
            cu = [0]
            for sq, _ in seqs:
                cu.append(cu[-1] + sq)
            pq = torch.randn((cu[-1], hq_p, HEAD_DIM), generator=g, device=dev,
                             dtype=torch.float32).to(torch.bfloat16)
            pout = torch.empty_like(pq)
            plse = torch.empty((hq_p, cu[-1]), dtype=torch.float32, device=dev)
            cu_t = torch.tensor(cu, dtype=torch.int32, device=dev)
            used = torch.tensor([n for _, n in seqs], dtype=torch.int32, device=dev)
            max_q = max(sq for sq, _ in seqs)
            flops = sum(prefill_flops(sq, n, n - sq, hq_p) for sq, n in seqs)

            def pp_call():
                fa.fa512_prefill_paged(pq, kp, vp, pt, cu_t, used, pout, plse, max_seqlen_q=max_q,
                                       stream=stream)

            for _ in range(max(3, args.warmup)):
                flush.zero_()
                pp_call()
            torch.cuda.synchronize()
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(args.steps)]
            cs = leg_sampler(dev)
            for e0, e1 in evs:
                flush.zero_()
                e0.record(stream)
                pp_call()
                e1.record(stream)
            torch.cuda.synchronize()
            leg_clocks = cs.stop()
            (t_pp,) = max_over_ranks([sum(e0.elapsed_time(e1) for e0, e1 in evs) / 1e3], dev)
            tf = job_rate(flops, args.steps, world, t_pp) / 1e12
            prefill_paged[name] = {
                "workload": "%d chunk(s) (rows, cached keys) %s over shuffled %d-key pages, "
                            "%d/%d heads, causal" % (len(seqs), seqs, PAGE, hq_p, hk_p),
                "value": tf, "unit": "TFLOP/s", "ms": t_pp / args.steps * 1e3,
                "flops_per_call": flops, "frac_of_measured_bf16": tf / world / peaks["bf16_tflops"],
                "l2": "flushed before every call", "clocks": leg_clocks}
            del kp, vp, pq, pout
        assert fa.fa512_device_status() == 0

    # ---- the local layers: heads of 256 dimensions over a 1,024-key window
    local256 = None
    if not args.no_prefill and not args.no_paged:
        L = LOCAL256
        lq = torch.randn((L["seqlen"], L["n_q_heads"], 256), generator=g, device=dev,
                         dtype=torch.float32).to(torch.bfloat16)
        lk = torch.randn((L["seqlen"], L["n_kv_heads"], 256), generator=g, device=dev,
                         dtype=torch.float32).to(torch.bfloat16)
        lv = torch.randn(lk.shape, generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
        lout = torch.empty_like(lq)
        llse = torch.empty((L["n_q_heads"], L["seqlen"]), dtype=torch.float32, device=dev)
        lflops = prefill_flops(L["seqlen"], L["seqlen"], 0, L["n_q_heads"], window=L["window"],
                               head_dim=256)

        def l_call():
            fa.fa512_prefill_d256(lq, lk, lv, lout, llse, window=L["window"], stream=stream)

        for _ in range(max(3, args.warmup)):
            flush.zero_()
            l_call()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        cs = leg_sampler(dev)
        for e0, e1 in evs:
            flush.zero_()
            e0.record(stream)
            l_call()
            e1.record(stream)
        torch.cuda.synchronize()
        leg_clocks = cs.stop()
        (t_l,) = max_over_ranks([sum(e0.elapsed_time(e1) for e0, e1 in evs) / 1e3], dev)
        tf = job_rate(lflops, args.steps, world, t_l) / 1e12
        local256 = {"workload": "local layer: %d tokens from 0, window %d, %d/%d heads, head dim 256, "
                                "causal" % (L["seqlen"], L["window"], L["n_q_heads"], L["n_kv_heads"]),
                    "value": tf, "unit": "TFLOP/s", "ms": t_l / args.steps * 1e3,
                    "flops_per_call": lflops, "frac_of_measured_bf16": tf / world / peaks["bf16_tflops"],
                    "l2": "flushed before every call", "clocks": leg_clocks}
        del lq, lk, lv, lout
        assert fa.fa512_device_status() == 0

    # ---- the full and MQA prefill configs (and the stress variant), each
    # timed on its own: one call per step, L2 flushed before every call
    prefill_legs = {}
    if not args.no_prefill and not args.no_big:
        for name, L in PREFILL_LEGS.items():
            if args.only_big and name not in args.only_big.split(","):
                continue
            bq = torch.randn((L["seqlen_q"], L["n_q_heads"], HEAD_DIM), generator=g, device=dev,
                             dtype=torch.float32).to(torch.bfloat16)
            bk = torch.randn((L["seqlen_k"], L["n_kv_heads"], HEAD_DIM), generator=g, device=dev,
                             dtype=torch.float32).to(torch.bfloat16)
            bv = torch.randn(bk.shape, generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
            if L["stress"]:
                bk[::64] *= 8          # every 64th key row x8 (exact in bf16)
            bout = torch.empty_like(bq)
            blse = torch.empty((L["n_q_heads"], L["seqlen_q"]), dtype=torch.float32, device=dev)
            flops = prefill_flops(L["seqlen_q"], L["seqlen_k"], L["q_offset"], L["n_q_heads"])

            def b_call():
                fa.fa512_prefill(bq, bk, bv, bout, blse, q_offset=L["q_offset"], causal=True,
                                 stream=stream)

            for _ in range(max(3, args.warmup)):
                flush.zero_()
                b_call()
            torch.cuda.synchronize()
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(args.steps)]
            cs = leg_sampler(dev)
            for e0, e1 in evs:
                flush.zero_()
                e0.record(stream)
                b_call()
                e1.record(stream)
            torch.cuda.synchronize()
            leg_clocks = cs.stop()
            (t_b,) = max_over_ranks([sum(e0.elapsed_time(e1) for e0, e1 in evs) / 1e3], dev)
            tf = job_rate(flops, args.steps, world, t_b) / 1e12
            ach = flops / (t_b / args.steps) / 1e12
            prefill_legs[name] = {
                "workload": "%d x %d causal prefill, %d/%d heads, d512, bf16 N(0,1)%s"
                            % (L["seqlen_q"], L["seqlen_k"], L["n_q_heads"], L["n_kv_heads"],
                               "; every 64th K row x8" if L["stress"] else ""),
                "value": tf, "unit": "TFLOP/s", "ms": t_b / args.steps * 1e3,
                "flops_per_call": flops,
                "target_ms_at_50pct_of_measured_burst": flops / (0.5 * peaks["bf16_tflops"] * 1e12) * 1e3,
                "roofline": {"kernel": "fa512::prefill_so::prefill_so_kernel<false>", "bound": "tensor",
                             "achieved": ach, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                             "frac": ach / peaks["bf16_tflops"],
                             "frac_of_sustained": ach / peaks["bf16_tflops_sustained"],
                             "peak_kind": "%s burst bf16 (MEASURED_PEAKS.json)" % peak_kind,
                             "traffic": recorded_traffic("prefill_so_kernel_" + name, pf_src)},
                "l2": "flushed before every call", "clocks": leg_clocks}
            del bq, bk, bv, bout, blse
        assert fa.fa512_device_status() == 0

    # ---- the decode shapes over an FP8 E4M3 cache, timed on their own
    decode_fp8 = None
    if not args.no_decode and not args.no_fp8:
        decode_fp8 = time_decode_fp8(args, fa, g, dev, stream, shapes, flush, world, peaks)
        assert fa.fa512_device_status() == 0

    # ---- paged decode of q_len tokens per sequence, timed on its own
    decode_q = None
    # (--decode-shapes selects main-loop shapes for profiling and skips this
    # leg unless --decode-q-batch asks for it)
    if not args.no_decode and (not args.decode_shapes or args.decode_q_batch is not None):
        b = args.decode_q_batch if args.decode_q_batch is not None else DECODE_Q_SHAPE["batch"]
        n, ql = DECODE_Q_SHAPE["kv_len"], DECODE_Q_SHAPE["q_len"]
        npg = (n + PAGE - 1) // PAGE
        gcpu = torch.Generator()
        gcpu.manual_seed(0x5EED + 6)
        kp = torch.randn((b * npg, PAGE, hk, HEAD_DIM), generator=g, device=dev,
                         dtype=torch.float32).to(torch.bfloat16)
        vp = torch.randn(kp.shape, generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
        pt = torch.randperm(b * npg, generator=gcpu).to(torch.int32).view(b, npg).to(dev)
        kl = torch.full((b,), n, dtype=torch.int32, device=dev)
        dq = torch.randn((b, ql, hq, HEAD_DIM), generator=g, device=dev,
                         dtype=torch.float32).to(torch.bfloat16)
        dout = torch.empty_like(dq)
        dlse = torch.empty((b, ql, hq), dtype=torch.float32, device=dev)
        ws = torch.empty(max(256, int(fa.load_library().fa512_decode_workspace_bytes_q(
            b, ql, hq, hk, PAGE, n, 0))), dtype=torch.uint8, device=dev)

        def dq_call():
            fa.fa512_decode_paged_q(dq, kp, vp, pt, kl, dout, dlse, max_kv_len=n, workspace=ws,
                                    stream=stream)

        for _ in range(max(3, args.warmup)):
            flush.zero_()
            dq_call()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        cs = leg_sampler(dev)
        for e0, e1 in evs:
            flush.zero_()
            e0.record(stream)
            dq_call()
            e1.record(stream)
        torch.cuda.synchronize()
        leg_clocks = cs.stop()
        (t_dq,) = max_over_ranks([sum(e0.elapsed_time(e1) for e0, e1 in evs) / 1e3], dev)
        dq_bytes = decode_bytes(b, n, hq, hk, ql)
        gbs = job_rate(dq_bytes, args.steps, world, t_dq) / 1e9
        decode_q = {"workload": "paged decode of %d tokens per sequence: batch %d x kv %d, "
                                "%d/%d heads, page %d, num_splits auto" % (ql, b, n, hq, hk, PAGE),
                    "value": gbs, "unit": "GB/s", "ms": t_dq / args.steps * 1e3,
                    "bytes_per_call": dq_bytes, "frac_of_measured_hbm": gbs / world / peaks["hbm_gbs"],
                    "l2": "flushed before every call", "clocks": leg_clocks}

    cpu = None
    if rank == 0 and world >= 1 and not args.no_cpu:
        f, dt, threads, desc = oracle_sample(budget_rows=args.ref_rows)
        cpu = {"value": f / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": desc, "seconds": dt, "plan": oracle_plan()}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_step / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": PREFILL_WORKLOAD + (DECODE_WORKLOAD if dec else ""),
                       "l2": "flushed (512 MiB write) before every step",
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "prefill_ms": t_pf / args.steps * 1e3,
            "decode": ({"value": dec_gbs, "unit": "GB/s", "ms": t_dec / args.steps * 1e3,
                        "bytes_per_step": dec_bytes} if dec else None),
            "roofline": roofline,
            "decode_roofline": decode_roofline,
            "decode_q": decode_q,
            "decode_fp8": decode_fp8,
            "prefill_paged": prefill_paged,
            "local256": local256,
            "prefill_full": prefill_legs.get("prefill_full"),
            "prefill_full_stress": prefill_legs.get("prefill_full_stress"),
            "prefill_mqa": prefill_legs.get("prefill_mqa"),
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": ((0 if args.no_prefill else 1) + 2 * len(dec)) * args.steps,
            "clocks": clocks,
            "wall_s_timed_region": wall,
            "device_status": status,
            "context": "pages: FA4 hd512 chunked prefill 302-336 TFLOP/s on GH200 "
                       "(44-49% of 686); not this hardware",
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ref-rows", type=int, default=24)
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-paged", action="store_true", help="skip the paged-prefill legs")
    ap.add_argument("--no-fp8", action="store_true", help="skip the FP8-cache decode leg")
    ap.add_argument("--no-big", action="store_true",
                    help="skip the full (20480^2, + stress) and MQA (49152^2) prefill legs")
    ap.add_argument("--only-big", default="",
                    help="comma list of big prefill legs to run (profiling), e.g. prefill_mqa")
    ap.add_argument("--decode-q-batch", type=int, default=None,
                    help="batch of the several-token decode leg (default 64; profiling a smaller case)")
    ap.add_argument("--no-prefill", action="store_true", help="decode only (profiling)")
    ap.add_argument("--decode-shapes", default="", help="comma list such as b64_kv28672")
    args = ap.parse_args()
    if args.warmup < 3:
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
