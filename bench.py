#!/usr/bin/env python
"""Decode-attention benchmark: µs per decode step and achieved HBM GB/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

One step is one gqa_decode call (one split-KV kernel launch, LSE merge included)
over the whole workload -- every sequence, every query head, one layer. The
default workload is the largest one that fits one GPU: ragged multi-token
decode (B=64, sq=4 causal, H=64, G=8, D=128, lengths uniform in [512, 32768] in
a 32768-token cache). Inputs are seeded synthetic N(0,1) bf16 tensors from the
synthetic/ generator.

value    = algorithmic bytes per step / device time per step (GB/s, all ranks);
           the K timed launches are enqueued behind a device-side spin, so the
           events time back-to-back device work, not the binding's call rate
e2e      = the same with the step's inputs copied from pinned host memory and its
           outputs copied back inside the timed region (inputs: Q, the lengths and
           the cache rows each (sequence, KV head) holds; a paged pool whole)
roofline = the split-KV kernel (the step's only launch): its average duration
           over the timed region, CUDA events on the launching stream,
           against the measured HBM copy bandwidth
cpu_baseline = the fp64 CPU oracle (test infrastructure) on the host cores,
           over a bounded sample of the workload's sequences
workloads = every other full-size decode workload (Llama-3-8B-shaped layer, MHA
           and MQA ends, long context at B = 1 and 4), timed in the same run by
           the same method (--workloads none|NAME,... changes the set)

Prefill workloads (--workload prefill_* / chunked_prefill_*) run gqa_prefill
instead and report TFLOP/s over the visible (causal) keys against the measured
bf16 tensor rate; a short chunk whose key ranges are split is two launches per
step (prefill kernel, then the combine). --fp8, --paged N and --append time the
other decode entry points on the same workloads.

Under torchrun (N > 1) every rank runs an independent replica of the workload
on its own GPU (the path has no exchange step); timing is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synthetic as syn  # noqa: E402

METRIC = "decode-attention µs/step and achieved HBM GB/s (% of GB300 peak) at 1 GPU"
DEFAULT_WORKLOAD = "ragged_sq4"
PROFILES = os.path.join(ROOT, "profiles")
KERNEL_SOURCES = [os.path.join(ROOT, "grouped_query_decode_gb300", "csrc", f) for f in
                  ("gqa_splitkv.cuh", "gqa_device.cuh", "gqa_common.h", "ptx.cuh", "gqa_launch_impl.cuh",
                   "api.cu")]


# ------------------------------------------------------------ accounting

def _percentiles_us(ms_list):
    """p10, median and p90 of per-call event times (ms), in microseconds."""
    if not ms_list:
        return None
    xs = sorted(ms_list)

    def at(f):
        # nearest rank on the sorted sample
        return xs[min(len(xs) - 1, max(0, int(round(f * (len(xs) - 1)))))] * 1e3

    return [at(0.10), at(0.50), at(0.90)]


def kv_bytes(G: int, D: int, lens, elem_bytes: int = 2) -> int:
    """K and V bytes one decode step must read: 2 (K and V) x sum_b T_b x G x D
    x element size -- the KV-cache sizing formula of "GQA analysis" (section
    "KV cache") for one layer, summed over the batch's actual lengths."""
    return 2 * int(np.sum(np.asarray(lens, dtype=np.int64))) * G * D * elem_bytes


def algorithmic_bytes(B: int, sq: int, H: int, G: int, D: int, lens) -> int:
    """Bytes a step must move at minimum: the valid K/V, Q in, O out (bf16),
    LSE out (fp32) and the lengths (int32). Tmax padding is not counted."""
    return kv_bytes(G, D, lens) + 2 * (B * sq * H * D * 2) + B * sq * H * 4 + 4 * B


def algorithmic_flops(sq: int, H: int, D: int, lens) -> int:
    """QK^T and PV multiply-adds: each query row does T_b*D of each ("keep query
    heads, cut KV heads", section "what shrinks and what does not": the score
    and weighted-sum counts carry no G), 2 flops per multiply-add."""
    return 4 * sq * H * D * int(np.sum(np.asarray(lens, dtype=np.int64)))


def visible_keys(sq: int, lens) -> int:
    """Keys all query rows of one head see: new token s of sequence b attends
    to positions t <= T_b - sq + s, i.e. max(0, T_b - sq + s + 1) keys."""
    total = 0
    for t in np.asarray(lens, dtype=np.int64):
        s = np.arange(sq, dtype=np.int64)
        total += int(np.maximum(0, t - sq + s + 1).sum())
    return total


def prefill_flops(H: int, D: int, sq: int, lens) -> int:
    """QK^T and PV over the visible (causal) keys only: 2 x 2 flops per key per
    head dimension element per query row."""
    return 4 * H * D * visible_keys(sq, lens)


def prefill_launches_per_step(B: int, sq: int, H: int, G: int, Tmax: int, sms: int) -> int:
    """Kernel launches one gqa_prefill call makes: the prefill kernel, plus the
    combine kernel when the library splits key ranges. It does that for short
    chunks whose pairs of 128-row tiles (B*G*ceil(tiles/2) items) cannot fill
    the SMs: splits = min(sms // items, key_tiles // 2) when 2*items <= sms,
    at most 32, or GQA_PREFILL_SPLITS when set."""
    rows = (H // G) * sq
    items = B * G * ((-(-rows // 128) + 1) // 2)
    splits = 1
    if 2 * items <= sms:
        splits = max(1, min(sms // items, -(-Tmax // 128) // 2))
    forced = int(os.environ.get("GQA_PREFILL_SPLITS", "0") or 0)
    if forced > 0:
        splits = forced
    return 2 if min(splits, 32) > 1 else 1


# --------------------------------------------------------------- helpers

def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def _code_of(text: str) -> str:
    """C/C++/CUDA source without its comments and blank lines, each line
    stripped: what the compiler sees of it (string literals in these files
    hold no comment markers)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*", "", ln).strip() for ln in text.splitlines())
    return "\n".join(ln for ln in lines if ln)


def _source_digest() -> str:
    """Hash of the kernel sources' code (comments left out, so that a comment
    edit does not orphan the ncu counters taken on the same code)."""
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(p, encoding="utf-8") as f:
            h.update(_code_of(f.read()).encode())
    return h.hexdigest()[:16]


def _ncu_traffic(workload: str):
    """DRAM bytes per launch of the split-KV kernel from the committed ncu
    summary of this exact workload and variant (e.g. "llama3_8b_layer+fp8"),
    if it was taken on the current kernel sources."""
    path = os.path.join(PROFILES, f"ncu_splitkv_{workload}.md")
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line and line.startswith("- "):
                k, v = line[2:].split(":", 1)
                vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_sources_sha256_16") != _source_digest():
        return None
    try:
        return int(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while work runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def aggregate_over_ranks(ms_per_step: float, bytes_per_rank: int, device=None):
    """Max of the per-step time over all ranks (the slowest rank sets the job's
    pace) and the whole-job throughput: every rank processed bytes_per_rank per
    step (weak scaling, independent replicas). Without an initialised process
    group this is the single-GPU case."""
    import torch
    import torch.distributed as dist
    ws = dist.get_world_size() if dist.is_available() and dist.is_initialized() else 1
    if ws > 1:
        t = torch.tensor([ms_per_step], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_per_step = float(t.item())
    return ms_per_step, ws * bytes_per_rank / (ms_per_step * 1e-3) / 1e9


# ----------------------------------------------------------- CPU oracle

def _cpu_model() -> str:
    """The host CPU's name from /proc/cpuinfo: "model name" (x86), else the
    Arm implementer and part numbers, else the machine type."""
    info = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if ":" in line:
                    key, val = line.split(":", 1)
                    info.setdefault(key.strip(), val.strip())
    except OSError:
        pass
    if info.get("model name"):
        return info["model name"]
    if "CPU part" in info:
        arm_parts = {"0xd4f": "Neoverse V2", "0xd40": "Neoverse V1", "0xd0c": "Neoverse N1",
                     "0xd49": "Neoverse N2"}
        part = info["CPU part"].lower()
        return f"Arm {arm_parts.get(part, 'part ' + part)} (implementer {info.get('CPU implementer', '?')})"
    import platform
    return platform.machine() or "unknown"


def time_oracle(cfg, q, k, v, lens, budget_s: float, max_reps: int | None = None):
    """Times the oracle (as it stands) over the whole step's rows, split over
    the host's cores; repeats the step until about budget_s of wall time."""
    import oracle
    threads = os.cpu_count() or 1
    orc = oracle.get()
    times = []
    t_all = time.perf_counter()
    while True:
        t0 = time.perf_counter()
        orc.gqa_decode(q, k, v, lens, cfg.scale, threads=threads)
        times.append(time.perf_counter() - t0)
        if max_reps is not None and len(times) >= max_reps:
            break
        if max_reps is None and time.perf_counter() - t_all >= budget_s:
            break
    return times, threads


def run_reference(args, cfg):
    """The reference arm: the fp64 CPU oracle, the only other implementation of
    this path there is, timed on the host cores over whole decode steps."""
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    q, k, v, lens = syn.make_inputs(cfg, tail_bits=syn.BF16_ZERO)
    if cfg in syn.PREFILL_CONFIGS:
        # A whole prefill takes the oracle minutes: each step is the bounded
        # sample of the CPU baseline (the last new tokens, every head).
        rates = []
        for _ in range(max(1, args.steps)):
            rate, threads, sample = time_oracle_prefill(cfg, q, k, v, lens, 0)
            rates.append(rate)
        value = statistics.median(rates)
        line = {
            "impl": "reference", "metric": "prefill attention TFLOP/s (causal keys only) at 1 GPU",
            "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": _config_dict(cfg, lens, l2_note="host memory"),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "sample": sample, "cpu_model": _cpu_model()},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }
        print(json.dumps(line), flush=True)
        return 0
    # Each step is the oracle over a bounded sample of the batch (the whole
    # batch where one step stays within the sample's budget).
    n = _oracle_sample(cfg, lens)
    q, k, v, lens = q[:n], k[:n], v[:n], lens[:n]
    nbytes = algorithmic_bytes(n, cfg.sq, cfg.H, cfg.G, cfg.D, lens)
    time_oracle(cfg, q, k, v, lens, 0, max_reps=max(1, args.warmup))
    times, threads = time_oracle(cfg, q, k, v, lens, 0, max_reps=args.steps)
    t = sum(times) / len(times)
    value = nbytes / t / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": _config_dict(cfg, lens, l2_note="host memory"),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"sequences 0..{n - 1} of {cfg.B} ({n * cfg.sq * cfg.H} query rows, "
                                   f"{nbytes} algorithmic bytes) per step, {args.steps} steps",
                         "seconds": sum(times), "cpu_model": _cpu_model()},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def _config_dict(cfg, lens, l2_note, append=False, paged=0, fp8=False):
    return {"workload": cfg.name + ("+append" if append else "") + (f"+paged{paged}" if paged else "")
            + ("+fp8" if fp8 else ""), "B": cfg.B, "sq": cfg.sq, "H": cfg.H, "G": cfg.G, "D": cfg.D,
            "Tmax": cfg.Tmax, "sum_T": int(np.sum(lens)), "scale": cfg.scale, "seed": cfg.seed,
            "inputs": "Q,K,V i.i.d. N(0,1) rounded to bf16", "l2": l2_note}


# ------------------------------------------------------------ GPU arm

# Full-size decode workloads timed in the same run as the headline line, each
# by the same method, into its "workloads" map (the headline's own workload is
# left out of the map). The tiny workload is launch-bound and not among them.
MAP_WORKLOADS = ("llama3_8b_layer", "long_ctx_b1", "long_ctx_b4", "mha_end", "mqa_end", "ragged_sq4")


def _variant_name(cfg, append=False, paged=0, fp8=False) -> str:
    return (cfg.name + ("+append" if append else "") + (f"+paged{paged}" if paged else "")
            + ("+fp8" if fp8 else ""))


class DecodeWorkload:
    """Device tensors of one decode workload (and entry-point variant) and its
    step: one call over the whole batch. The K/V caches rotate over enough
    copies that their footprint is at least 4x L2, so no step finds its K/V
    left in L2 by the step before."""

    def __init__(self, cfg, dev, append=False, paged=0, fp8=False, keep_host=False):
        import torch

        import grouped_query_decode_gb300 as gq

        self.gq = gq
        self.cfg, self.dev = cfg, dev
        self.append, self.paged, self.fp8 = append, paged, fp8
        self.name = _variant_name(cfg, append, paged, fp8)
        q, k, v, lens = syn.make_inputs(cfg, tail_bits=syn.BF16_ZERO)
        self.lens = lens
        self.nbytes = algorithmic_bytes(cfg.B, cfg.sq, cfg.H, cfg.G, cfg.D, lens)
        self.flops = algorithmic_flops(cfg.sq, cfg.H, cfg.D, lens)

        def to_dev(bits):
            return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)

        self.to_dev = to_dev
        props = torch.cuda.get_device_properties(dev)
        self.l2 = int(getattr(props, "L2_cache_size", 126 * 2 ** 20))
        self.cache_bytes = 2 * k.nbytes
        self.copies = copies = max(2, math.ceil(4 * self.l2 / self.cache_bytes))
        self.dq = to_dev(q)
        self.dl = torch.from_numpy(lens).to(dev)
        self.out = torch.empty(cfg.B, cfg.sq, cfg.H, cfg.D, dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty(cfg.B, cfg.sq, cfg.H, dtype=torch.float32, device=dev)
        self.host_q, self.host_kv = q, None
        if fp8:
            # The same caches as e4m3 codes with one fp32 scale per 64-token block.
            kc, ksc = syn.fp8_cache(k, lens, tail_code=0)
            vc, vsc = syn.fp8_cache(v, lens, tail_code=0)
            self.sets = [(torch.from_numpy(kc).to(dev), torch.from_numpy(vc).to(dev),
                          torch.from_numpy(ksc).to(dev), torch.from_numpy(vsc).to(dev))
                         for _ in range(copies)]
            self.nbytes += (kv_bytes(cfg.G, cfg.D, lens, elem_bytes=1)    # 1-byte codes ...
                            - kv_bytes(cfg.G, cfg.D, lens)                  # ... instead of bf16
                            + 2 * 4 * int(sum(-(-int(t) // 64) for t in lens)) * cfg.G)  # block scales
            if keep_host:
                self.host_kv = (kc, vc, ksc, vsc)
        elif paged:
            # The same logical caches laid out in pages, one paged copy per
            # rotation slot, each with its own block table.
            self.sets = []
            for c in range(copies):
                kp, vp, table = syn.paginate(k, v, lens, paged, seed=cfg.seed + 100 + c,
                                             fill_bits=syn.BF16_ZERO)
                self.sets.append((to_dev(kp), to_dev(vp), torch.from_numpy(table).to(dev)))
                if c == 0 and keep_host:
                    self.host_kv = (kp, vp, table)
            self.nbytes += sum(-(-int(t) // paged) for t in lens) * 4     # block-table entries read
        else:
            self.sets = [(to_dev(k), to_dev(v)) for _ in range(copies)]
            if keep_host:
                self.host_kv = (k, v)
        if append:
            # Fused append: each step also writes the sq new tokens' K/V rows.
            self.dkn = to_dev(syn.normal_bf16(cfg.seed, 11, (cfg.B, cfg.sq, cfg.G, cfg.D)))
            self.dvn = to_dev(syn.normal_bf16(cfg.seed, 12, (cfg.B, cfg.sq, cfg.G, cfg.D)))
            self.nbytes += 2 * 2 * (cfg.B * cfg.sq * cfg.G * cfg.D * 2)   # new rows read + written
        self.host_bf16 = (k, v) if keep_host else None

    def l2_note(self) -> str:
        return (f"inputs larger than L2: {self.copies} rotating K/V copies of "
                f"{self.cache_bytes >> 20} MiB vs {self.l2 >> 20} MiB L2")

    def call(self, stream, kv):
        gq, cfg = self.gq, self.cfg
        if self.fp8:
            kc, vc, ks, vs = kv
            gq.gqa_decode_fp8(self.dq, kc, vc, ks, vs, self.dl, cfg.scale, self.out, self.lse, stream=stream)
        elif self.paged:
            kp, vp, tb = kv
            gq.gqa_decode_paged(self.dq, kp, vp, tb, self.dl, cfg.scale, self.out, self.lse, stream=stream)
        elif self.append:
            gq.gqa_decode_append(self.dq, self.dkn, self.dvn, kv[0], kv[1], self.dl, cfg.scale, self.out,
                                 self.lse, stream=stream)
        else:
            gq.gqa_decode(self.dq, kv[0], kv[1], self.dl, cfg.scale, self.out, self.lse, stream=stream)

    def step(self, i, stream):
        self.call(stream, self.sets[i % self.copies])


def e2e_copy_pairs(dkv, hkv, lens, fp8=False):
    """(device view, host view) pairs an end-to-end step copies for a
    contiguous cache: the rows each (sequence, KV head) holds, since the rows
    past a sequence's length are never read and so are not inputs of the step
    (for fp8 block scales [B, G, blocks]: the 64-token blocks those rows
    touch). Runs of sequences whose rows fill the cache are one copy."""
    pairs = []
    B = len(lens)
    for d, h in zip(dkv, hkv):
        per_block = 64 if (fp8 and h.dim() == 3) else 1
        G, full = h.shape[1], h.shape[2]
        rows = [-(-int(t) // per_block) for t in lens]
        b = 0
        while b < B:
            if rows[b] >= full:
                e = b
                while e < B and rows[e] >= full:
                    e += 1
                pairs.append((d[b:e], h[b:e]))
                b = e
                continue
            if rows[b]:
                pairs += [(d[b, g, :rows[b]], h[b, g, :rows[b]]) for g in range(G)]
            b += 1
    return pairs


def _spin(host_us_per_call: float, calls: int):
    """Keeps the stream busy on the device for about as long as the host takes
    to enqueue `calls` more calls (capped at 0.2 s), so that the calls
    enqueued behind it run back to back: the events around them then time
    the device's work, not the binding's call rate. Spins on the SM clock
    (torch's sleep kernel), counted at 2.1 GHz, at least the maximum SM clock."""
    import torch
    us = min(2e5, 20.0 + 1.25 * host_us_per_call * calls)
    torch.cuda._sleep(int(us * 2100))


def time_steps(step, steps: int, warmup: int, dev, stream, gpu_index: int, ws: int):
    """W untimed warm-up steps, then exactly `steps` timed steps on `stream`
    between two CUDA events, bracketed by barrier + synchronize; then the same
    number (at most 200) of calls each between its own events. The host
    enqueues each timed run behind a device-side spin (_spin). nvidia-smi
    samples the clocks meanwhile. Returns (ms per step, per-call ms list,
    clocks summary)."""
    import torch
    import torch.distributed as dist

    import grouped_query_decode_gb300 as gq

    host_us = []
    for i in range(max(3, warmup)):
        t0 = time.perf_counter()
        step(i)
        host_us.append((time.perf_counter() - t0) * 1e6)
    torch.cuda.synchronize(dev)
    assert gq.gqa_decode_check_error(stream) == gq.GQA_OK
    call_us = statistics.median(host_us[1:]) if len(host_us) > 1 else host_us[0]

    sampler = ClockSampler(gpu_index)
    sampler.start()
    time.sleep(0.15)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t_wall0 = time.perf_counter()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    _spin(call_us, steps)
    e0.record(stream)
    for i in range(steps):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    if ws > 1:
        dist.barrier()
    t_wall = time.perf_counter() - t_wall0
    ms_total = e0.elapsed_time(e1)
    # keep sampling the same work a little longer if the region was short
    t_tail = time.perf_counter()
    i = 0
    while time.perf_counter() - t_tail < max(0.0, 0.6 - t_wall):
        step(i)
        i += 1
        if i % 256 == 0:
            torch.cuda.synchronize(dev)
    torch.cuda.synchronize(dev)
    sampler.stop()
    clocks = sampler.summary()
    clocks["window"] = "timed region" if t_wall >= 0.6 else "timed region + untimed tail of the same step"

    # Per-call durations: events around each call, enqueued behind a spin too.
    n_calls = min(steps, 200) if steps > 0 else 0
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n_calls)]
    _spin(call_us, n_calls)
    for i, (a, b) in enumerate(evs):
        a.record(stream)
        step(i)
        b.record(stream)
    torch.cuda.synchronize(dev)
    assert gq.gqa_decode_check_error(stream) == gq.GQA_OK
    return ms_total / steps, [a.elapsed_time(b) for a, b in evs], clocks, call_us


def _roofline_entry(wl, ms_step: float, call_ms, peak: float) -> dict:
    achieved = wl.nbytes / (ms_step * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "kernel": "gqa_splitkv_kernel", "duration_us": ms_step * 1e3,
            "per_call_us": statistics.mean(call_ms) * 1e3 if call_ms else None,
            "per_call_p10_p50_p90_us": _percentiles_us(call_ms),
            "algorithmic_bytes_per_launch": wl.nbytes,
            "traffic": _ncu_traffic(wl.name)}


def _oracle_sample(cfg, lens, flop_budget: float = 2e10) -> int:
    """Sequences of the oracle's bounded sample: the first n of the batch, n
    as large as keeps one sampled step within flop_budget (about half a second
    of the fp64 oracle on 16 host cores)."""
    per_seq = [4 * cfg.sq * cfg.H * cfg.D * int(t) for t in lens]
    n, acc = 0, 0
    for f in per_seq:
        if n > 0 and acc + f > flop_budget:
            break
        acc += f
        n += 1
    return n


def run_gpu(args, cfg):
    import torch
    import torch.distributed as dist

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=dev)
    stream = torch.cuda.current_stream(dev)
    peak, peak_kind = _peaks()
    variant = dict(append=args.append, paged=args.paged, fp8=args.fp8)

    wl = DecodeWorkload(cfg, dev, keep_host=True, **variant)
    ms_step, call_ms, clocks, host_call_us = time_steps(lambda i: wl.step(i, stream), args.steps, args.warmup,
                                                        dev, stream, local, ws)
    ms_step, value = aggregate_over_ranks(ms_step, wl.nbytes, device=dev)
    roof = _roofline_entry(wl, ms_step, call_ms, peak)
    roof.update({
        "peak_kind": peak_kind,
        "duration": f"average over the {args.steps} launches of the timed region (CUDA events on the "
                    "launching stream; one launch per step; the launches are enqueued behind a device-side "
                    "spin, so no step waits for the host)",
        "per_call": f"{len(call_ms)} calls each between its own events (also enqueued behind a spin)",
        "host_us_per_call": host_call_us,
    })

    # End to end through the public API: inputs from pinned host memory to the
    # device, the call, outputs back, every step, all inside the timed region.
    q = wl.host_q
    hq = torch.from_numpy(q.view(np.int16)).view(torch.bfloat16).pin_memory()
    hl = torch.from_numpy(wl.lens).pin_memory()
    if args.fp8:
        hkv = [torch.from_numpy(x).pin_memory() for x in wl.host_kv]
    elif args.paged:
        kp, vp, table = wl.host_kv
        hkv = [torch.from_numpy(kp.view(np.int16)).view(torch.bfloat16).pin_memory(),
               torch.from_numpy(vp.view(np.int16)).view(torch.bfloat16).pin_memory(),
               torch.from_numpy(table).pin_memory()]
    else:
        hkv = [torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory() for x in wl.host_kv]
    dkv = wl.sets[0]
    copies = list(zip(dkv, hkv)) if args.paged else e2e_copy_pairs(dkv, hkv, wl.lens, fp8=args.fp8)
    ho = torch.empty(wl.out.shape, dtype=torch.bfloat16).pin_memory()
    hlse = torch.empty(wl.lse.shape, dtype=torch.float32).pin_memory()
    if args.append:
        hkn = wl.dkn.cpu().pin_memory()
        hvn = wl.dvn.cpu().pin_memory()

    def e2e_step():
        wl.dq.copy_(hq, non_blocking=True)
        for d, h in copies:
            d.copy_(h, non_blocking=True)
        wl.dl.copy_(hl, non_blocking=True)
        if args.append:
            wl.dkn.copy_(hkn, non_blocking=True)
            wl.dvn.copy_(hvn, non_blocking=True)
        wl.call(stream, dkv)
        ho.copy_(wl.out, non_blocking=True)
        hlse.copy_(wl.lse, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize(dev)
    if ws > 1:
        dist.barrier()
    e2e_steps = max(3, min(args.steps, 20))
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    b.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms, e2e_value = aggregate_over_ranks(a.elapsed_time(b) / e2e_steps, wl.nbytes, device=dev)
    h2d = hq.nbytes + hl.nbytes + sum(h.nbytes for _, h in copies)
    if args.append:
        h2d += hkn.nbytes + hvn.nbytes
    d2h = ho.nbytes + hlse.nbytes
    del hq, hl, hkv, ho, hlse, dkv, copies

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        k, v = wl.host_bf16
        n = _oracle_sample(cfg, wl.lens)
        sub_bytes = algorithmic_bytes(n, cfg.sq, cfg.H, cfg.G, cfg.D, wl.lens[:n])
        times, threads = time_oracle(cfg, q[:n], k[:n], v[:n], wl.lens[:n], args.cpu_budget_s)
        tc = statistics.median(times)
        cpu = {"value": sub_bytes / tc / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
               "sample": (f"sequences 0..{n - 1} of {cfg.B} (every head and new token: "
                          f"{n * cfg.sq * cfg.H} query rows, {sub_bytes} algorithmic bytes) x "
                          f"{len(times)} repetitions, median"),
               "seconds": sum(times), "cpu_model": _cpu_model()}
    config = _config_dict(cfg, wl.lens, l2_note=wl.l2_note(), **variant)
    nbytes, flops, name = wl.nbytes, wl.flops, wl.name
    del wl
    torch.cuda.empty_cache()

    # The other full-size decode workloads, same variant, same method.
    names = [n for n in MAP_WORKLOADS if n != cfg.name] if args.workloads == "default" else \
        ([] if args.workloads == "none" else [n for n in args.workloads.split(",") if n])
    workloads = {}
    for wname in names:
        wcfg = syn.config_by_name(wname)
        w = DecodeWorkload(wcfg, dev, **variant)
        w_ms, w_calls, w_clocks, _ = time_steps(lambda i: w.step(i, stream), args.steps, args.warmup,
                                                 dev, stream, local, ws)
        w_ms, w_value = aggregate_over_ranks(w_ms, w.nbytes, device=dev)
        entry = _roofline_entry(w, w_ms, w_calls, peak)
        workloads[w.name] = {
            "us_per_step": w_ms * 1e3, "value": w_value, "unit": "GB/s", "frac": entry["frac"],
            "per_call_p10_p50_p90_us": entry["per_call_p10_p50_p90_us"],
            "algorithmic_bytes_per_step": w.nbytes, "traffic": entry["traffic"],
            "gpu_launches": args.steps,
            "config": {k: getattr(wcfg, k) for k in ("B", "sq", "H", "G", "D", "Tmax")} |
                      {"sum_T": int(np.sum(w.lens)), "l2": w.l2_note()},
            "clocks": w_clocks,
        }
        del w
        torch.cuda.empty_cache()

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "us_per_step": ms_step * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": config,
            "query_tokens_per_s": ws * cfg.B * cfg.sq / (ms_step * 1e-3),
            "tflops": ws * flops / (ms_step * 1e-3) / 1e12,
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "GB/s",
                    "us_per_step": e2e_ms * 1e3,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "h2d": ("Q, the lengths and the whole paged pool with its block table" if args.paged else
                            "Q, the lengths and the cache rows each (sequence, KV head) holds"
                            + (" with their block scales" if args.fp8 else "")
                            + (" and the new tokens' K/V" if args.append else "")),
                    "d2h": "out and lse"},
            "gpu_launches": args.steps,
            "clocks": clocks,
            "workloads": workloads,
            "workloads_note": ("every other full-size decode workload, timed in this run by the same method "
                               f"({args.warmup} warm-up and {args.steps} timed steps, CUDA events, inputs "
                               "larger than L2); value in GB/s of algorithmic bytes, frac of the same peak"),
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


# ------------------------------------------------------- prefill GPU arm

def _tensor_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


def time_oracle_prefill(cfg, q, k, v, lens, budget_s: float, rows_tokens: int = 16):
    """The oracle (as it stands) on a bounded sample of a prefill: the last
    `rows_tokens` new tokens of every sequence (all heads), which see the most
    keys. Returns (TFLOP/s, threads, description)."""
    import oracle
    threads = os.cpu_count() or 1
    orc = oracle.get()
    n = min(rows_tokens, cfg.sq)
    qs = np.ascontiguousarray(q[:, cfg.sq - n:])
    flops = 4 * cfg.H * cfg.D * visible_keys(n, lens)
    times = []
    t_all = time.perf_counter()
    while True:
        t0 = time.perf_counter()
        orc.gqa_decode(qs, k, v, lens, cfg.scale, threads=threads)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_all >= budget_s:
            break
    tc = statistics.median(times)
    return flops / tc / 1e12, threads, (f"last {n} new tokens of each of the {cfg.B} sequences "
                                        f"({cfg.B * n * cfg.H} query rows), {len(times)} repetitions, median")


def run_gpu_prefill(args, cfg):
    import torch
    import torch.distributed as dist

    import grouped_query_decode_gb300 as gq

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=dev)

    q, k, v, lens = syn.make_inputs(cfg, tail_bits=syn.BF16_ZERO)
    flops = prefill_flops(cfg.H, cfg.D, cfg.sq, lens)
    nbytes = algorithmic_bytes(cfg.B, cfg.sq, cfg.H, cfg.G, cfg.D, lens)

    def to_dev(bits):
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)

    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2 ** 20))
    cache_bytes = 2 * k.nbytes
    copies = max(2, math.ceil(4 * l2 / cache_bytes))
    dq = to_dev(q)
    dl = torch.from_numpy(lens).to(dev)
    dks = [to_dev(k) for _ in range(copies)]
    dvs = [to_dev(v) for _ in range(copies)]
    out = torch.empty(cfg.B, cfg.sq, cfg.H, cfg.D, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(cfg.B, cfg.sq, cfg.H, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(i):
        c = i % copies
        gq.gqa_prefill(dq, dks[c], dvs[c], dl, cfg.scale, out, lse, stream=stream)

    kernel_ms, call_ms, clocks, _ = time_steps(step, args.steps, args.warmup, dev, stream, local, ws)
    ms_step, _ = aggregate_over_ranks(kernel_ms, nbytes, device=dev)
    value = ws * flops / (ms_step * 1e-3) / 1e12
    launches = prefill_launches_per_step(cfg.B, cfg.sq, cfg.H, cfg.G, cfg.Tmax,
                                         torch.cuda.get_device_properties(dev).multi_processor_count)
    n_calls = len(call_ms)
    achieved = flops / (kernel_ms * 1e-3) / 1e12
    peak, peak_kind = _tensor_peak()

    # End to end: inputs from pinned host memory, outputs back, every step.
    hq = torch.from_numpy(q.view(np.int16)).view(torch.bfloat16).pin_memory()
    hk = torch.from_numpy(k.view(np.int16)).view(torch.bfloat16).pin_memory()
    hv = torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).pin_memory()
    hl = torch.from_numpy(lens).pin_memory()
    ho = torch.empty(out.shape, dtype=torch.bfloat16).pin_memory()
    hlse = torch.empty(lse.shape, dtype=torch.float32).pin_memory()

    def e2e_step():
        dq.copy_(hq, non_blocking=True)
        dks[0].copy_(hk, non_blocking=True)
        dvs[0].copy_(hv, non_blocking=True)
        dl.copy_(hl, non_blocking=True)
        gq.gqa_prefill(dq, dks[0], dvs[0], dl, cfg.scale, out, lse, stream=stream)
        ho.copy_(out, non_blocking=True)
        hlse.copy_(lse, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize(dev)
    if ws > 1:
        dist.barrier()
    e2e_steps = max(3, min(args.steps, 20))
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    b.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms, _ = aggregate_over_ranks(a.elapsed_time(b) / e2e_steps, nbytes, device=dev)

    if rank == 0:
        cpu = None
        if ws == 1 and not args.no_cpu_baseline:
            t_cpu = time.perf_counter()
            rate, threads, sample = time_oracle_prefill(cfg, q, k, v, lens, args.cpu_budget_s)
            cpu = {"value": rate, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": sample,
                   "seconds": time.perf_counter() - t_cpu, "cpu_model": _cpu_model()}
        line = {
            "metric": "prefill attention TFLOP/s (causal keys only) at 1 GPU", "value": value,
            "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_step, "us_per_step": ms_step * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": _config_dict(cfg, lens, l2_note=f"{copies} rotating K/V copies of "
                                                      f"{cache_bytes >> 20} MiB vs {l2 >> 20} MiB L2"),
            "query_tokens_per_s": ws * cfg.B * cfg.sq / (ms_step * 1e-3),
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak, "traffic": None, "peak_kind": peak_kind,
                         "kernel": "gqa_prefill_kernel", "duration_us": kernel_ms * 1e3,
                         "duration": f"average step over the {args.steps} steps of the timed region "
                                     "(CUDA events on the launching stream; "
                                     + ("one launch per step)" if launches == 1 else
                                        "two launches per step: the prefill kernel over split key "
                                        "ranges, then the combine kernel)"),
                         "launches_per_step": launches,
                         "per_call_us": statistics.mean(call_ms) * 1e3 if call_ms else None,
                         "per_call_p10_p50_p90_us": _percentiles_us(call_ms),
                         "per_call": f"{n_calls} calls each bracketed by its own events",
                         "algorithmic_flops_per_launch": flops},
            "cpu_baseline": cpu,
            "e2e": {"value": ws * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                    "us_per_step": e2e_ms * 1e3,
                    "h2d_bytes_per_step": hq.nbytes + hk.nbytes + hv.nbytes + hl.nbytes,
                    "d2h_bytes_per_step": ho.nbytes + hlse.nbytes},
            "gpu_launches": args.steps * launches,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=[c.name for c in syn.CONFIGS + syn.PREFILL_CONFIGS],
                    help="a decode workload, or a prefill workload (timed on gqa_prefill)")
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--cpu-budget-s", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--paged", type=int, default=0, metavar="PAGE_SIZE",
                    help="time gqa_decode_paged on the same caches split into pages of this size")
    ap.add_argument("--fp8", action="store_true",
                    help="time gqa_decode_fp8 on the same caches as e4m3 codes with block scales")
    ap.add_argument("--append", action="store_true",
                    help="time gqa_decode_append (new K/V rows written in the same launch)")
    ap.add_argument("--workloads", default="default",
                    help="decode workloads also timed into the line's 'workloads' map: 'default' (every "
                         "other full-size decode workload), 'none', or a comma-separated list of names")
    args = ap.parse_args(argv)
    cfg = syn.config_by_name(args.workload)
    if args.impl == "reference":
        return run_reference(args, cfg)
    if cfg in syn.PREFILL_CONFIGS:
        return run_gpu_prefill(args, cfg)
    return run_gpu(args, cfg)


if __name__ == "__main__":
    sys.exit(main())
