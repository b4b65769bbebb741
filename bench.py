#!/usr/bin/env python3
"""Throughput of the Engram layer prefill (hash -> gather -> project -> gate/add).

Default workload: 4 x 4096 Zipf(1.1) tokens with 5% image (DEAD) spans,
compressed vocabulary 99092, a 48,004,402-row table (12.67 GB of E4M3+E8M0
rows) from base 2,000,000, hidden 5120, 4 residual streams, wkv [6144, 25600].

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One JSON line is printed by rank 0.  A "step" is one pass of the whole layer
over one batch of 16384 tokens.  Timing: CUDA events on the launching stream
around every step; the L2 cache is flushed before every step, outside the
events (a 512 MB write, then a 256 MB read so that no dirty line is left to
write back inside the step).  Under torchrun every rank runs its own batch (no
collective on the data path, weak scaling) and the slowest rank's time is
used.  ``--impl reference`` times the CPU oracle on a bounded sample of the
same workload instead (rank 0 only).

Side phases, reported next to the headline: hash + gather on the 65,536-token
microbench batch, decode steps, and the same table kept in pinned host memory
(zero-copy gather over NVLink-C2C, and the prefetch pipeline).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Engram layer tokens/s (hash+gather+gate) at T=16k; gather HBM GB/s vs peak"
GATHER_BYTES_PER_TOKEN = 4 + 24 * 264 + 24 * 256 * 2   # raw id + 24 rows + bf16 e = 18,628 B
# the sources each profiled kernel is built from: a traffic figure is used
# only while the hash of its kernel's sources matches the one it was taken with
KERNEL_SOURCES = {
    "project2_kernel": ["project.cu", "engram_internal.h"],
    "project2_kernel_unfused": ["project.cu", "engram_internal.h"],
    "project8_kernel_unfused": ["project.cu", "engram_internal.h"],
    "gather_ldgsts_kernel": ["gather.cu", "hash_device.cuh", "engram_internal.h"],
    "gather_ldgsts_kernel_ids": ["gather.cu", "hash_device.cuh", "engram_internal.h"],
    "hash_prefill_kernel": ["hash.cu", "hash_device.cuh", "engram_internal.h"],
    "hash_commit_kernel": ["hash.cu", "hash_device.cuh", "engram_internal.h"],
    "gates_kernel": ["gate.cu", "engram_internal.h"],
    "gate_add_kernel": ["gate.cu", "engram_internal.h"],
    "conv_prep_kernel": ["shortconv.cu", "engram_internal.h"],
    "conv_add_kernel": ["shortconv.cu", "engram_internal.h"],
    "conv_state_kernel": ["shortconv.cu", "engram_internal.h"],
    "gather_ldgsts_kernel_microbench": ["gather.cu", "hash_device.cuh", "engram_internal.h"],
    "gather_ldgsts_kernel_microbench_fused": ["gather.cu", "hash_device.cuh", "engram_internal.h"],
    "gather_ldgsts_kernel_fp8": ["gather.cu", "hash_device.cuh", "engram_internal.h"],
    "gather_rows_bf16_kernel": ["gather_bf16.cu", "hash_device.cuh", "engram_internal.h"],
}


def GATE_BYTES_PER_TOKEN(hc: int, hidden: int) -> int:
    """Gate + residual add: h read and written (bf16), v read, the partial sums read, the mask."""
    return 2 * hc * hidden * 2 + hidden * 2 + hc * (hidden // 256) * 16 + 1


def CONV_BYTES_PER_TOKEN(hc: int, hidden: int) -> int:
    """Short convolution + residual: h read and written (bf16), v and the gates read once."""
    return 2 * hc * hidden * 2 + hidden * 2 + hc * 4


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=700)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="prefill")
    p.add_argument("--e2e-steps", type=int, default=30)
    p.add_argument("--micro-steps", type=int, default=30, help="steps of the hash+gather microbench phase")
    p.add_argument("--decode-steps", type=int, default=200, help="steps of the decode phase")
    p.add_argument("--conv-steps", type=int, default=30, help="steps of the short-convolution layer phase")
    p.add_argument("--fp8-steps", type=int, default=200, help="steps of the block-FP8 projection layer phase")
    p.add_argument("--generic-steps", type=int, default=30,
                   help="steps of the Engram-27B-shaped layer phase (bf16 rows of 80, hidden 2560)")
    p.add_argument("--fullscale-passes", type=int, default=2,
                   help="timed passes over the 131,072-token full-scale sequence (101 GB table; 0 skips it)")
    p.add_argument("--host-steps", type=int, default=20,
                   help="steps of the host-resident table phase (0 skips it and its pinned allocation)")
    p.add_argument("--cpu-sample", type=int, default=8192, help="tokens of the oracle CPU baseline sample")
    p.add_argument("--ref-sample", type=int, default=128, help="tokens per reference-arm step")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--sustained-s", type=float, default=3.0,
                   help="seconds of back-to-back layer steps after the timed region (projection under the power cap)")
    p.add_argument("--plain-launch", action="store_true",
                   help="launch the fused kernels without the cooperative attribute (for ncu; GPU must be exclusive)")
    return p.parse_args()


def workload_desc(w):
    return (f"{w.name}: {w.n_seqs} x {w.seq_len} Zipf(1.1) tokens, {int(w.dead_frac * 100)}% DEAD spans, "
            f"V_raw {w.v_raw} -> V {w.v}, 24 primes above {w.base_rows}, hidden {w.hidden}, hc {w.hc}, "
            f"wkv [6144, {(w.hc + 1) * w.hidden}]")


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def sources_hash(files, read=None) -> str:
    """Hash of the given kernel sources (read(name) -> bytes; the working tree by default)."""
    h = hashlib.sha256()
    for f in files:
        if read is None:
            with open(os.path.join(ROOT, "hashed_gram_conditional_gb300", "csrc", f), "rb") as fh:
                h.update(fh.read())
        else:
            h.update(read(f))
    return h.hexdigest()[:16]


def profiled_traffic():
    """Per-launch DRAM bytes from the committed ncu summary, for the kernels
    whose sources still hash to the values the counters were taken with."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return {}
    with open(path) as f:
        d = json.load(f)
    out = {}
    for name, entry in d.get("kernels", {}).items():
        files = KERNEL_SOURCES.get(name)
        if files is not None and entry.get("sources_hash") == sources_hash(files):
            out[name] = entry["bytes_per_launch"]
    return out


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling around a timed region.

    Samples every `interval_ms` with nvidia-smi's own timestamp; stop(t0, t1)
    keeps only the samples taken between the wall-clock times t0 and t1 (the
    timed region), and says how many that was."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str, interval_ms: int = 10):
        self.gpu_id = gpu_id
        self.interval_ms = interval_ms
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-lms", str(self.interval_ms), "-i", self.gpu_id], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    @staticmethod
    def _epoch(stamp: str):
        import datetime
        try:
            return datetime.datetime.strptime(stamp.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def stop(self, t0=None, t1=None):
        """Summary of the samples; with t0, t1 (time.time()) only those inside
        [t0, t1], widened by 50 ms steps (up to 250 ms) while none falls inside."""
        out = self._summary(t0, t1)
        pad = 0.0
        while t0 is not None and out["samples"] == 0 and pad < 0.25:
            pad += 0.05
            out = self._summary(t0 - pad, t1 + pad)
            out["window_widened_ms"] = round(pad * 1e3)
        return out

    def _summary(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        if self.proc.poll() is None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        total = 0
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 10:
                continue
            total += 1
            if t0 is not None:
                ts = self._epoch(parts[0])
                if ts is None or ts < t0 or ts > t1:
                    continue
            try:
                sm.append(float(parts[2]))
                smax.append(float(parts[3]))
                power.append(float(parts[4]))
            except ValueError:
                continue
            for n, v in zip(names, parts[6:10]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        out = {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
               "power_w_max": max(power) if power else None, "reasons": sorted(reasons), "samples": len(sm),
               "interval_ms": self.interval_ms}
        if t0 is not None:
            out["samples_outside_region"] = total - len(sm)
        return out


# ------------------------------------------------------------------------- ranks


def rank_seed(base_seed: int, rank: int) -> int:
    """Each replica draws its own batch (weak scaling, no shared data)."""
    return base_seed + rank


def reduce_max(x: float, world: int, device) -> float:
    """Largest value over ranks (the slowest rank's time)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_value(tokens_per_step: int, steps: int, world: int, max_total_s: float) -> float:
    """Whole-job tokens/s: every rank processed tokens_per_step per step."""
    return world * tokens_per_step * steps / max_total_s


# ------------------------------------------------------------------------- inputs


def make_inputs(w, seed, dev):
    import torch
    import hashed_gram_conditional_gb300 as eg
    from workloads import layer_weights, prefill_batch, residual_bits, token_map

    tm = token_map(w.v_raw, w.v, w.seed)
    lay = eg.build_layout(w.v, w.base_rows, [w.layer_id], pad_id=int(tm[0]), expected_vocab=w.v)
    total = lay.total_rows(0)
    table = torch.empty(total * eg.ROW_BYTES, dtype=torch.uint8, device=dev)
    eg.engram_fill_synthetic_table(table, total, w.seed)
    lw = layer_weights(w)

    def bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

    wkv = bf16(lw.wkv_bits)
    layer = eg.EngramLayer(lay, 0, table, torch.from_numpy(tm).to(dev), eg.engram_pack_wkv(wkv),
                           torch.from_numpy(lw.q_w).to(dev), torch.from_numpy(lw.k_w).to(dev))
    del wkv
    b = prefill_batch(w, seed=seed)
    h_bits = residual_bits(len(b.raw_ids), w.hc, w.hidden, seed)
    return dict(tm=tm, lay=lay, layer=layer, lw=lw, batch=b, h_bits=h_bits, bf16=bf16)


# ------------------------------------------------------------------------- our arm


def run_ours(args, rank, world, local):
    import torch
    import torch.distributed as dist
    import hashed_gram_conditional_gb300 as eg
    from workloads import WORKLOADS

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if args.plain_launch:
        eg.set_kernel_options(plain_launch=1)
    w = WORKLOADS[args.workload]
    inp = make_inputs(w, rank_seed(w.seed, rank), dev)
    layer, b = inp["layer"], inp["batch"]
    T = len(b.raw_ids)
    raw = torch.from_numpy(b.raw_ids).to(dev)
    cu = torch.from_numpy(b.cu_seqlens).to(dev)
    h = inp["bf16"](inp["h_bits"])
    h0 = h.clone()
    hist = torch.full((w.n_seqs, 3), inp["lay"].pad_id, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)

    b_ = layer._buffers(T, dev)

    def step(ev=None):
        # one pass of the whole layer; events between the stage launches when timing
        if ev is not None:
            ev[0].record(stream)
        eg.engram_hash_gather(layer.layout, 0, raw, cu, layer.token_map, layer.table, hist, b_["e"], b_["mask"],
                              None, status)
        if ev is not None:
            ev[1].record(stream)
        eg.engram_project_gate(b_["e"], layer.wkv_packed, h, layer.q_w, layer.k_w, b_["mask"], layer.eps,
                               layer.clamp, layer.score_scale, None, b_["work"], status)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} during warm-up")

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    props = torch.cuda.get_device_properties(dev)
    gpu_id = f"GPU-{props.uuid}" if getattr(props, "uuid", None) is not None else str(local)
    sampler = ClockSampler(gpu_id)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)  # let the sampler's first reading land
    epoch0 = time.time()
    wall0 = time.perf_counter()
    for k in range(args.steps):
        flush()
        step(events[k])
    torch.cuda.synchronize()
    wall1 = time.perf_counter()
    epoch1 = time.time()
    if world > 1:
        dist.barrier()
    time.sleep(0.05)  # the sampler's last readings of the region
    clocks = sampler.stop(epoch0, epoch1)
    st = int(status.item())

    def ms(k, i, j):
        return events[k][i].elapsed_time(events[k][j])

    step_ms = [ms(k, 0, 2) for k in range(args.steps)]
    stage = {name: [ms(k, i, i + 1) for k in range(args.steps)]
             for i, name in enumerate(["hash_gather", "project_gate"])}
    total_s = reduce_max(sum(step_ms) / 1e3, world, dev)

    # ---- end to end: host buffers through the public layer API.  Each step
    # copies its raw ids, cu_seqlens and residual h from pinned host memory
    # and reads the updated h back; the copies of step k+1 and k-1 run on
    # their own streams while step k computes (three buffer slots: with two,
    # one slot's copy-in, compute and copy-out would have to fit in two steps).
    e2e = None
    if args.e2e_steps > 0:
        e2e = e2e_pipeline(args, b, h0, layer, hist, status, dev, world)

    # side phases, reported next to the headline at N = 1 only (under
    # torchrun every rank would otherwise pin host memory and allocate the
    # full-scale table at once)
    side = world == 1
    hgg = hash_gather_gate_bench(args, w, inp, layer, flush, dev) if side and args.micro_steps > 0 else None
    micro = microbench(args, w, inp, layer, flush, dev) if side and args.micro_steps > 0 else None
    dec = decode_bench(args, w, inp, layer, flush, dev) if side and args.decode_steps > 0 else None
    conv = conv_bench(args, w, inp, layer, flush, dev) if side and args.conv_steps > 0 else None
    fp8 = fp8_bench(args, w, inp, layer, flush, dev) if side and args.fp8_steps > 0 else None
    gen = generic_bench(args, w, flush, dev) if side and args.generic_steps > 0 else None
    host = host_table_bench(args, w, inp, layer, flush, dev, statistics.mean(step_ms)) \
        if side and args.host_steps > 0 else None
    full = fullscale_bench(args, inp, layer, dev) if side and args.fullscale_passes > 0 else None
    # last, so that the heat of a seconds-long loop does not reach the other legs
    sus = sustained_loop(args.sustained_s, step, flush, gpu_id) if side and args.sustained_s > 0 else None

    if rank != 0:
        return None

    peaks, peak_src = load_peaks()
    traffic = profiled_traffic()
    timed_s = wall1 - wall0
    if micro is not None:
        micro["frac"] = micro["gather_gbs"] / peaks["hbm_gbs"]
        micro["peak_gbs"] = peaks["hbm_gbs"]
        micro["uniform_control"]["frac"] = micro["uniform_control"]["gather_gbs"] / peaks["hbm_gbs"]
    if hgg is not None:
        hgg["gate_frac_hbm"] = hgg["gate_gbs"] / peaks["hbm_gbs"]
        hgg["hash_gather_frac_hbm"] = hgg["hash_gather_gbs"] / peaks["hbm_gbs"]
    if full is not None and "hash_gather_gbs" in full:
        full["hash_gather_frac_hbm"] = full["hash_gather_gbs"] / peaks["hbm_gbs"]
    if gen is not None:
        gen["hash_gather_frac_hbm"] = gen["hash_gather_gbs"] / peaks["hbm_gbs"]
    if dec is not None:
        dec["wkv_frac_hbm"] = dec["wkv_gbs"] / peaks["hbm_gbs"]
    if fp8 is not None:
        # fp8 dense tensor peak: the measured bf16 figure times the nominal fp8 / bf16 ratio (4.5 / 2.25)
        fp8_sust = fp8["timed_s"] >= 2.0
        pk = 2.0 * (peaks["bf16_tflops_sustained"] if fp8_sust else peaks["bf16_tflops"])
        fp8["roofline"] = {"bound": "tensor", "kernel": "project8_kernel<unfused> (tcgen05 kind::mxf8f6f4)",
                           "achieved": fp8["project_tflops"], "peak": pk, "unit": "TFLOP/s",
                           "frac": fp8["project_tflops"] / pk,
                           "peak_source": f"{peak_src} bf16_tflops{'_sustained' if fp8_sust else ''} x 2 "
                                          "(nominal fp8 / bf16 dense ratio)",
                           "traffic": traffic.get("project8_kernel_unfused")}
    if conv is not None:
        conv["conv_frac_hbm"] = conv["conv_gbs"] / peaks["hbm_gbs"]
        conv["traffic_conv_add"] = traffic.get("conv_add_kernel")
    # A timed region of 2 s or more of back-to-back steps runs under the power
    # cap like the driver's sustained GEMM loop; shorter ones compare to burst.
    sustained = timed_s >= 2.0
    tf_peak = peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"]
    flops = 2.0 * T * 6144 * (w.hc + 1) * w.hidden
    proj_s = statistics.mean(stage["project_gate"]) / 1e3
    gat_s = statistics.mean(stage["hash_gather"]) / 1e3
    roof = {"bound": "tensor",
            "kernel": "project2_kernel<fused> (CTA-pair tcgen05 wkv GEMM, gate and residual in the epilogue)",
            "achieved": flops / proj_s / 1e12, "peak": tf_peak, "unit": "TFLOP/s",
            "frac": flops / proj_s / 1e12 / tf_peak, "frac_vs_burst": flops / proj_s / 1e12 / peaks["bf16_tflops"],
            "traffic": traffic.get("project2_kernel"),
            "algorithmic_per_launch": f"{flops:.4g} FLOP (2*T*6144*{(w.hc + 1) * w.hidden}, T={T})",
            "peak_source": f"{peak_src} bf16_tflops{'_sustained' if sustained else ''}"}
    gbytes = GATHER_BYTES_PER_TOKEN * T
    gather_kernel = "gather_ldgsts_kernel"
    roof_g = {"bound": "hbm", "kernel": "gather_ldgsts_kernel<HashedRows> (hash fused into the gather) + the history "
                                        "commit", "achieved": gbytes / gat_s / 1e9,
              "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": gbytes / gat_s / 1e9 / peaks["hbm_gbs"],
              "traffic": traffic.get(gather_kernel),
              "algorithmic_per_launch": f"{gbytes} B ({GATHER_BYTES_PER_TOKEN} B/token, T={T})",
              "peak_source": f"{peak_src} hbm_gbs"}
    # the gather half of the metric, nested in the roofline record: the fused
    # hash + gather inside the timed step and the 65,536-token microbench
    roof["hash_gather"] = {
        "in_step": {k: roof_g[k] for k in ("kernel", "achieved", "peak", "unit", "frac", "traffic",
                                            "algorithmic_per_launch", "peak_source")},
    }
    roof["hash_gather"]["in_step"]["ms"] = gat_s * 1e3
    if micro is not None:
        Tm = micro["algorithmic_bytes"] // GATHER_BYTES_PER_TOKEN
        for key, kern in (("microbench_fused", "fused"), ("microbench", "gather")):
            if key == "microbench_fused" and "fused_gather_gbs" not in micro:
                continue
            gbs = micro["fused_gather_gbs"] if key == "microbench_fused" else micro["gather_gbs"]
            roof["hash_gather"][key] = {
                "kernel": ("gather_ldgsts_kernel<HashedRows> (hash fused into the gather)" if kern == "fused"
                           else "gather_ldgsts_kernel<IdRows> (engram_gather_dequant after engram_hash)"),
                "tokens": Tm, "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": gbs / peaks["hbm_gbs"],
                "algorithmic_per_launch": f"{micro['algorithmic_bytes']} B ({GATHER_BYTES_PER_TOKEN} B/token)",
                "traffic": traffic.get(f"{gather_kernel}_microbench" if kern == "gather"
                                       else f"{gather_kernel}_microbench_fused"),
                "uniform_tokens_frac": (micro["uniform_control"]["fused_gather_gbs"] if kern == "fused"
                                        else micro["uniform_control"]["gather_gbs"]) / peaks["hbm_gbs"]
                if (kern == "gather" or "fused_gather_gbs" in micro["uniform_control"]) else None,
                "peak_source": f"{peak_src} hbm_gbs"}
    if full is not None and "hash_gather_gbs" in full:
        roof["hash_gather"]["full_scale"] = {
            "kernel": "gather_ldgsts_kernel<HashedRows>, 101.4 GB table, 16,384-token chunks",
            "achieved": full["hash_gather_gbs"], "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": full["hash_gather_gbs"] / peaks["hbm_gbs"]}
    if gen is not None:
        roof["hash_gather"]["generic_27b_shape"] = {
            "kernel": "gather_rows_bf16_kernel<hashed> + the history commit", "achieved": gen["hash_gather_gbs"],
            "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": gen["hash_gather_gbs"] / peaks["hbm_gbs"],
            "traffic": traffic.get("gather_rows_bf16_kernel")}
    if dec is not None:
        roof["decode_wkv"] = {"kernel": "projection at 256 tokens (wkv streamed from HBM)",
                              "achieved": dec["wkv_gbs"], "peak": peaks["hbm_gbs"], "unit": "GB/s",
                              "frac": dec["wkv_gbs"] / peaks["hbm_gbs"], "step_ms": dec.get("step_ms"),
                              "project_gate_ms": dec.get("project_gate_ms")}
    roof["frac_vs_sustained"] = flops / proj_s / 1e12 / peaks["bf16_tflops_sustained"]
    if clocks.get("sm_mhz"):
        roof["sm_mhz_median_timed"] = clocks["sm_mhz"]
    if sus is not None:
        tf = flops / (sus["project_gate_ms"] / 1e3) / 1e12
        roof["sustained_loop"] = {
            "seconds": sus["wall_s"], "steps": sus["steps"], "project_gate_ms": sus["project_gate_ms"],
            "achieved": tf, "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s",
            "frac": tf / peaks["bf16_tflops_sustained"], "frac_vs_burst": tf / peaks["bf16_tflops"],
            "sm_mhz_median": sus["clocks"].get("sm_mhz"), "power_w_max": sus["clocks"].get("power_w_max"),
            "reasons": sus["clocks"].get("reasons"), "clock_samples": sus["clocks"].get("samples"),
            "tflops_per_ghz": (tf / (sus["clocks"]["sm_mhz"] / 1e3)) if sus["clocks"].get("sm_mhz") else None,
            "peak_source": f"{peak_src} bf16_tflops_sustained (sm_mhz_median "
                           f"{peaks.get('clocks_under_load', {}).get('sm_mhz_median')})"}
    out = {
        "metric": METRIC,
        "value": aggregate_value(T, args.steps, world, total_s),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": total_s / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded Zipf tokens, SplitMix64 table, N(0,0.02) wkv, N(0,1) residual)",
        "config": {"workload": workload_desc(w), "tokens_per_step": T, "parallelism": f"replicas x{world}",
                   "l2": "flushed before every step (512 MB write, then 256 MB read; outside the timed events)"},
        "stages_ms": {k: statistics.mean(v) for k, v in stage.items()},
        "roofline": roof,
        "roofline_gather": roof_g,
        "hash_gather_gate": hgg,
        "microbench_hash_gather": micro,
        "decode_step": dec,
        "short_conv_layer": conv,
        "fp8_layer": fp8,
        "generic_27b_shape": gen,
        "fullscale": full,
        "host_table": host,
        "gpu_launches": args.steps * 3,
        "clocks": clocks,
        "e2e": e2e,
        "wall_s_timed": wall1 - wall0,
        "device_status": st,
    }
    if world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(w, inp, args.cpu_sample)
    return out


def sustained_loop(seconds, step, flush, gpu_id):
    """Layer steps back to back for ``seconds`` after the timed region, with
    the SM clocks sampled meanwhile: the projection's rate under the power
    cap, comparable with the driver's sustained GEMM peak (also a
    seconds-long loop).  Same step and L2 flush as the timed region."""
    import torch
    sampler = ClockSampler(gpu_id, interval_ms=50)
    sampler.start()
    time.sleep(0.3)
    e0 = time.time()
    evs = []
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        batch = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(50)]
        for ev in batch:
            flush()
            step(ev)
        torch.cuda.synchronize()
        evs.extend(batch)
    wall = time.perf_counter() - t0
    clocks = sampler.stop(e0, time.time())
    return {"steps": len(evs), "wall_s": wall,
            "project_gate_ms": statistics.mean(ev[1].elapsed_time(ev[2]) for ev in evs),
            "hash_gather_ms": statistics.mean(ev[0].elapsed_time(ev[1]) for ev in evs),
            "step_ms": statistics.mean(ev[0].elapsed_time(ev[2]) for ev in evs), "clocks": clocks}


def e2e_pipeline(args, b, h0, layer, hist, status, dev, world):
    """Host-to-host layer prefill through EngramLayer.prefill, copies overlapped with compute."""
    import torch
    raw_h = torch.from_numpy(b.raw_ids).pin_memory()
    cu_h = torch.from_numpy(b.cu_seqlens).pin_memory()
    h_host = h0.cpu().pin_memory()
    T = raw_h.numel()
    slots = [dict(raw=torch.empty(T, dtype=torch.int32, device=dev),
                  cu=torch.empty(cu_h.numel(), dtype=torch.int64, device=dev),
                  h=torch.empty_like(h0),
                  out=torch.empty_like(h_host).pin_memory(),
                  copied=torch.cuda.Event(), computed=torch.cuda.Event(), drained=torch.cuda.Event())
             for _ in range(3)]
    s_in, s_comp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def run(steps, t_start=None, t_end=None, marks=None):
        if t_start is not None:
            t_start.record(s_in)
        for k in range(steps):
            sl = slots[k % len(slots)]
            s_in.wait_event(sl["drained"])          # the slot's previous result has left the device
            with torch.cuda.stream(s_in):
                sl["raw"].copy_(raw_h, non_blocking=True)
                sl["cu"].copy_(cu_h, non_blocking=True)
                sl["h"].copy_(h_host, non_blocking=True)
                sl["copied"].record(s_in)
            s_comp.wait_event(sl["copied"])
            with torch.cuda.stream(s_comp):
                layer.prefill(sl["raw"], sl["cu"], sl["h"], hist, status)
                sl["computed"].record(s_comp)
            s_out.wait_event(sl["computed"])
            with torch.cuda.stream(s_out):
                sl["out"].copy_(sl["h"], non_blocking=True)
                sl["drained"].record(s_out)
                if marks is not None:
                    marks[k].record(s_out)
        if t_end is not None:
            t_end.record(s_out)

    run(3)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(args.e2e_steps)]
    run(args.e2e_steps, e0, e1, marks)
    torch.cuda.synchronize()
    tot = reduce_max(e0.elapsed_time(e1) / 1e3, world, dev)
    gaps = [marks[k - 1].elapsed_time(marks[k]) for k in range(1, len(marks))]
    h2d = raw_h.numel() * 4 + cu_h.numel() * 8 + h_host.numel() * 2
    return {"value": aggregate_value(T, args.e2e_steps, world, tot), "unit": "tokens/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(h_host.numel() * 2),
            "steps": args.e2e_steps, "ms_per_step": tot / args.e2e_steps * 1e3,
            "ms_between_results_median": statistics.median(gaps) if gaps else None,
            "ms_between_results_max": max(gaps) if gaps else None,
            "api": "EngramLayer.prefill on a compute stream; pinned host inputs copied in and the updated residual "
                   "copied out on two copy streams, three buffer slots, so step k+1's input and step k-1's output "
                   "move while step k computes"}


class L2Flush:
    """Empties L2 between steps: a 512 MB write evicts everything, then a
    256 MB read replaces the written lines with clean ones.  A write alone
    leaves ~126 MB of dirty lines whose write-back then lands inside the next
    step (measured on GB300: +12 us on the 256-token projection)."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
        self.r = torch.ones(64 * 1024 * 1024, dtype=torch.int32, device=dev)

    def __call__(self):
        self.w.zero_()
        self.r.max()


def hash_gather_gate_bench(args, w, inp, layer, flush, dev):
    """The layer without the wkv GEMM (the metric's hash + gather + gate): the
    fused hash + gather, then the gate and residual add from partial sums and
    v produced once, outside the timed region, by the projection."""
    import torch
    import hashed_gram_conditional_gb300 as eg

    b = inp["batch"]
    T = len(b.raw_ids)
    raw = torch.from_numpy(b.raw_ids).to(dev)
    cu = torch.from_numpy(b.cu_seqlens).to(dev)
    h = inp["bf16"](inp["h_bits"])
    e, mask = eg.engram_hash_gather(layer.layout, 0, raw, cu, layer.token_map, layer.table)
    partials, v = eg.engram_project(e, layer.wkv_packed, h, layer.q_w, layer.k_w)
    stream = torch.cuda.current_stream(dev)

    def run(ev=None):
        if ev is not None:
            ev[0].record(stream)
        eg.engram_hash_gather(layer.layout, 0, raw, cu, layer.token_map, layer.table, None, e, mask)
        if ev is not None:
            ev[1].record(stream)
        eg.engram_gate_add(partials, v, h, mask, layer.eps, layer.clamp, layer.score_scale)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(3):
        flush()
        run()
    n = args.micro_steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
    for k in range(n):
        flush()
        run(evs[k])
    torch.cuda.synchronize()
    step = statistics.mean(ev[0].elapsed_time(ev[2]) for ev in evs) / 1e3
    hg = statistics.mean(ev[0].elapsed_time(ev[1]) for ev in evs) / 1e3
    gate = statistics.mean(ev[1].elapsed_time(ev[2]) for ev in evs) / 1e3
    gb = GATE_BYTES_PER_TOKEN(w.hc, w.hidden) * T
    return {"workload": f"{w.name} batch ({T} tokens), L2 flushed before every step", "steps": n,
            "tokens_per_s": T / step, "ms_per_step": step * 1e3, "hash_gather_ms": hg * 1e3, "gate_ms": gate * 1e3,
            "hash_gather_gbs": GATHER_BYTES_PER_TOKEN * T / hg / 1e9, "gate_gbs": gb / gate / 1e9,
            "gate_algorithmic_bytes": gb, "kernels": "gather_ldgsts_kernel<HashedRows> + gate_add_kernel"}


def fullscale_bench(args, inp, layer, dev):
    """The full-scale configuration: a 384,006,168-row (101.4 GB) table from
    base 16,000,000 and one 131,072-token sequence prefilled in 8 chunks of
    16,384 with the history carried; the same projection weights."""
    import torch
    import hashed_gram_conditional_gb300 as eg
    from workloads import WORKLOADS, prefill_batch, token_map

    wf = WORKLOADS["fullscale"]
    tm = token_map(wf.v_raw, wf.v, wf.seed)
    lay = eg.build_layout(wf.v, wf.base_rows, [wf.layer_id], pad_id=int(tm[0]), expected_vocab=wf.v)
    total = lay.total_rows(0)
    free, _ = torch.cuda.mem_get_info(dev)
    if free < total * eg.ROW_BYTES + (6 << 30):
        return {"skipped": f"needs {total * eg.ROW_BYTES / 1e9:.1f} GB free, {free / 1e9:.1f} GB available"}
    table = torch.empty(total * eg.ROW_BYTES, dtype=torch.uint8, device=dev)
    eg.engram_fill_synthetic_table(table, total, wf.seed)
    fl = eg.EngramLayer(lay, 0, table, torch.from_numpy(tm).to(dev), layer.wkv_packed, layer.q_w, layer.k_w)
    b = prefill_batch(wf)
    T = len(b.raw_ids)
    C = T // wf.chunks
    raw = torch.from_numpy(b.raw_ids).to(dev)
    cu = torch.tensor([0, C], dtype=torch.int64, device=dev)
    h = inp["bf16"](inp["h_bits"][:C])
    hist = torch.full((1, 3), lay.pad_id, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    buf = fl._buffers(C, dev)
    stream = torch.cuda.current_stream(dev)

    def one_pass(evs=None):
        hist.fill_(lay.pad_id)
        for c in range(wf.chunks):
            if evs is not None:
                evs[c][0].record(stream)
            eg.engram_hash_gather(lay, 0, raw[c * C:(c + 1) * C], cu, fl.token_map, table, hist, buf["e"],
                                  buf["mask"], None, status)
            if evs is not None:
                evs[c][1].record(stream)
            eg.engram_project_gate(buf["e"], fl.wkv_packed, h, fl.q_w, fl.k_w, buf["mask"], fl.eps, fl.clamp,
                                   fl.score_scale, None, buf["work"], status)
            if evs is not None:
                evs[c][2].record(stream)

    one_pass()
    torch.cuda.synchronize()
    res = []
    for _ in range(args.fullscale_passes):
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(wf.chunks)]
        one_pass(evs)
        torch.cuda.synchronize()
        res.append(evs)
    tot = sum(ev[c][0].elapsed_time(ev[c][2]) for ev in res for c in range(wf.chunks)) / 1e3
    hg = sum(ev[c][0].elapsed_time(ev[c][1]) for ev in res for c in range(wf.chunks)) / 1e3
    n_tok = T * args.fullscale_passes
    out = {"workload": f"fullscale: 1 x {T} Zipf(1.1) tokens in {wf.chunks} chunks of {C}, history carried, "
                       f"{total * eg.ROW_BYTES / 1e9:.1f} GB table (primes above {wf.base_rows})",
           "passes": args.fullscale_passes, "tokens_per_s": n_tok / tot, "ms_per_chunk": tot / (wf.chunks *
                                                                                                 args.fullscale_passes) * 1e3,
           "hash_gather_ms_per_chunk": hg / (wf.chunks * args.fullscale_passes) * 1e3,
           "hash_gather_gbs": GATHER_BYTES_PER_TOKEN * n_tok / hg / 1e9, "device_status": int(status.item()),
           "note": "chunks run back to back (no L2 flush; the table is 101 GB, so rows come from HBM)"}
    del fl, table
    torch.cuda.empty_cache()
    return out


def microbench(args, w, inp, layer, flush, dev):
    """Hash + gather only on the 65,536-token microbench workload (same table)."""
    import torch
    import hashed_gram_conditional_gb300 as eg
    from workloads import WORKLOADS, prefill_batch

    wm = WORKLOADS["microbench"]
    if (wm.base_rows, wm.v, wm.v_raw, wm.layer_id, wm.seed) != (w.base_rows, w.v, w.v_raw, w.layer_id, w.seed):
        return None
    bm = prefill_batch(wm)
    T = len(bm.raw_ids)
    raw = torch.from_numpy(bm.raw_ids).to(dev)
    cu = torch.from_numpy(bm.cu_seqlens).to(dev)
    rows = torch.empty((T, 24), dtype=torch.int32, device=dev)
    mask = torch.empty(T, dtype=torch.uint8, device=dev)
    e = torch.empty((T, 6144), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)

    def run(ev=None):
        if ev is not None:
            ev[0].record(stream)
        eg.engram_hash(layer.layout, 0, raw, cu, layer.token_map, None, rows, mask)
        if ev is not None:
            ev[1].record(stream)
        eg.engram_gather_dequant(layer.table, layer.total_rows, rows, e)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(3):
        flush()
        run()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.micro_steps)]
    for k in range(args.micro_steps):
        flush()
        run(evs[k])
    torch.cuda.synchronize()
    step = statistics.mean(ev[0].elapsed_time(ev[2]) for ev in evs) / 1e3
    gat = statistics.mean(ev[1].elapsed_time(ev[2]) for ev in evs) / 1e3
    gbytes = GATHER_BYTES_PER_TOKEN * T
    # control: uniformly random tokens (no Zipf reuse of hot rows in L2)
    g = np.random.default_rng(wm.seed + 77)
    raw = torch.from_numpy(g.integers(0, wm.v_raw, size=T).astype(np.int32)).to(dev)
    for _ in range(3):
        flush()
        run()
    evu = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.micro_steps)]
    for k in range(args.micro_steps):
        flush()
        run(evu[k])
    torch.cuda.synchronize()
    gat_u = statistics.mean(ev[1].elapsed_time(ev[2]) for ev in evu) / 1e3

    # the product path: hash fused into the gather (one kernel), Zipf then uniform tokens
    def fused(raw_ids, ev=None):
        if ev is not None:
            ev[0].record(stream)
        eg.engram_hash_gather(layer.layout, 0, raw_ids, cu, layer.token_map, layer.table, None, e, mask)
        if ev is not None:
            ev[1].record(stream)

    fused_s = {}
    for name, raw_ids in (("zipf", torch.from_numpy(bm.raw_ids).to(dev)), ("uniform", raw)):
        for _ in range(3):
            flush()
            fused(raw_ids)
        evf = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.micro_steps)]
        for k in range(args.micro_steps):
            flush()
            fused(raw_ids, evf[k])
        torch.cuda.synchronize()
        fused_s[name] = statistics.mean(ev[0].elapsed_time(ev[1]) for ev in evf) / 1e3
    return {"workload": f"microbench: 1 x {T} Zipf(1.1) tokens, same 12.67 GB table", "steps": args.micro_steps,
            "hash_gather_tokens_per_s": T / step, "hash_ms": (step - gat) * 1e3, "gather_ms": gat * 1e3,
            "gather_gbs": gbytes / gat / 1e9, "algorithmic_bytes": gbytes,
            "fused_hash_gather_ms": fused_s["zipf"] * 1e3, "fused_gather_gbs": gbytes / fused_s["zipf"] / 1e9,
            "fused_tokens_per_s": T / fused_s["zipf"],
            "uniform_control": {"tokens": "uniform over the raw vocabulary", "gather_ms": gat_u * 1e3,
                                "gather_gbs": gbytes / gat_u / 1e9,
                                "fused_hash_gather_ms": fused_s["uniform"] * 1e3,
                                "fused_gather_gbs": gbytes / fused_s["uniform"] / 1e9}}


def decode_bench(args, w, inp, layer, flush, dev):
    """Decode steps: 256 sequences of the decode workload, one token each, over the bench's table."""
    import torch
    import hashed_gram_conditional_gb300 as eg
    from workloads import WORKLOADS, decode_workload

    wd = WORKLOADS["decode"]
    if (wd.v, wd.v_raw, wd.hidden, wd.hc) != (w.v, w.v_raw, w.hidden, w.hc):
        return None
    n = args.decode_steps
    dw = decode_workload(wd, n_steps=n + 3)
    B = wd.n_seqs
    hist = torch.full((B, 3), layer.layout.pad_id, dtype=torch.int32, device=dev)
    eg.engram_hash(layer.layout, 0, torch.from_numpy(dw.prefix.raw_ids).to(dev),
                   torch.from_numpy(dw.prefix.cu_seqlens).to(dev), layer.token_map, hist)
    steps = torch.from_numpy(dw.steps).to(dev)
    slots = torch.arange(B, dtype=torch.int32, device=dev)
    rows = torch.empty((B, 24), dtype=torch.int32, device=dev)
    mask = torch.empty(B, dtype=torch.uint8, device=dev)
    e = torch.empty((B, 6144), dtype=torch.bfloat16, device=dev)
    h = torch.randn((B, wd.hc, wd.hidden), device=dev).to(torch.bfloat16)
    work = eg.project_gate_workspace(B, wd.hidden, wd.hc, dev)
    stream = torch.cuda.current_stream(dev)

    def run(k, ev=None, fused=True):
        if ev is not None:
            ev[0].record(stream)
        if fused:
            eg.engram_hash_gather_step(layer.layout, 0, steps[k], slots, layer.token_map, layer.table, hist, e, mask)
        else:
            eg.engram_hash_step(layer.layout, 0, steps[k], slots, layer.token_map, hist, rows, mask)
        if ev is not None:
            ev[1].record(stream)
        if not fused:
            eg.engram_gather_dequant(layer.table, layer.total_rows, rows, e)
        if ev is not None:
            ev[2].record(stream)
        eg.engram_project_gate(e, layer.wkv_packed, h, layer.q_w, layer.k_w, mask, layer.eps, layer.clamp,
                               layer.score_scale, None, work)
        if ev is not None:
            ev[3].record(stream)

    def timed(fused):
        for k in range(3):
            flush()
            run(k, fused=fused)
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n)]
        for k in range(n):
            flush()
            run(3 + k, evs[k], fused=fused)
        torch.cuda.synchronize()
        return evs

    def mean_ms(evs, i, j):
        return statistics.mean(ev[i].elapsed_time(ev[j]) for ev in evs)

    # the separate hash step and gather first (for the split), then the fused
    # step from the same start; both advance the histories through the same steps
    evs = timed(False)
    hist.fill_(layer.layout.pad_id)
    eg.engram_hash(layer.layout, 0, torch.from_numpy(dw.prefix.raw_ids).to(dev),
                   torch.from_numpy(dw.prefix.cu_seqlens).to(dev), layer.token_map, hist)
    evf = timed(True)
    step = mean_ms(evf, 0, 3) / 1e3
    proj = mean_ms(evf, 2, 3) / 1e3
    wkv_bytes = 6144 * (wd.hc + 1) * wd.hidden * 2
    out = {"workload": f"decode: {B} sequences x 1 token, histories from U[0, 8192] prefixes, table of the "
                       f"{w.name} workload", "steps": n,
           "step_ms": step * 1e3, "steps_per_s": 1 / step, "tokens_per_s": B / step,
           "hash_gather_ms": mean_ms(evf, 0, 1), "project_gate_ms": proj * 1e3, "wkv_gbs": wkv_bytes / proj / 1e9,
           "kernels": "engram_hash_gather_step (hash + history roll + gather in one kernel), engram_project_gate",
           "separate_calls": {"step_ms": mean_ms(evs, 0, 3), "hash_step_ms": mean_ms(evs, 0, 1),
                              "gather_ms": mean_ms(evs, 1, 2), "project_gate_ms": mean_ms(evs, 2, 3)}}
    out["graph"] = decode_graph_timing(layer, steps, slots, hist, h, n, flush, stream)
    if args.fp8_steps <= 0:
        if not args.no_cpu_baseline:
            out["cpu_baseline"] = decode_cpu_baseline(w, inp, dw, 10)
        return out

    # The same steps with block-FP8 wkv: rows gathered as stored, block-scaled projection.
    w8p, sfb = fp8_weights(w, inp, dev)
    hist.fill_(layer.layout.pad_id)
    eg.engram_hash(layer.layout, 0, torch.from_numpy(dw.prefix.raw_ids).to(dev),
                   torch.from_numpy(dw.prefix.cu_seqlens).to(dev), layer.token_map, hist)
    e8 = torch.empty((B, 6144), dtype=torch.uint8, device=dev)
    sfa = torch.empty((48, eg.sf_cols(B)), dtype=torch.int32, device=dev)

    def run8(k, ev=None):
        if ev is not None:
            ev[0].record(stream)
        eg.engram_hash_gather_step_fp8(layer.layout, 0, steps[k], slots, layer.token_map, layer.table, hist, e8,
                                       sfa, mask)
        if ev is not None:
            ev[1].record(stream)
            ev[2].record(stream)
        eg.engram_project_gate_fp8(e8, sfa, w8p, sfb, h, layer.q_w, layer.k_w, mask, layer.eps, layer.clamp,
                                   layer.score_scale, None, work)
        if ev is not None:
            ev[3].record(stream)

    for k in range(3):
        flush()
        run8(k)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n)]
    for k in range(n):
        flush()
        run8(3 + k, evs[k])
    torch.cuda.synchronize()
    step8 = statistics.mean(ev[0].elapsed_time(ev[3]) for ev in evs) / 1e3
    proj8 = statistics.mean(ev[2].elapsed_time(ev[3]) for ev in evs) / 1e3
    wkv8_bytes = 6144 * (wd.hc + 1) * wd.hidden * (1 + 1 / 32)
    if not args.no_cpu_baseline:
        out["cpu_baseline"] = decode_cpu_baseline(w, inp, dw, 10)
    out["fp8"] = {"workload": "the same steps with block-FP8 wkv (E4M3, E8M0 per 32 of k), rows gathered as stored",
                  "step_ms": step8 * 1e3, "tokens_per_s": B / step8,
                  "hash_gather_ms": statistics.mean(ev[0].elapsed_time(ev[1]) for ev in evs),
                  "project_gate_ms": proj8 * 1e3, "wkv_gbs": wkv8_bytes / proj8 / 1e9}
    return out


def decode_graph_timing(layer, steps, slots, hist, h, n, flush, stream):
    """The layer's decode step captured as a CUDA graph (EngramLayer.decode_graph)
    against eager EngramLayer.decode calls: device time per step (L2 flushed,
    CUDA events) and wall-clock time per step of n steps issued back to back,
    which includes the host's launch work."""
    import torch

    B = slots.numel()
    graph = layer.decode_graph(B, hist, h)
    graph.slots.copy_(slots)
    n_avail = steps.shape[0]

    def eager(k):
        layer.decode(steps[k % n_avail], slots, hist, h)

    def replay(k):
        graph.raw_ids.copy_(steps[k % n_avail])
        graph.replay()

    def wall(fn):
        for k in range(3):
            fn(k)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for k in range(n):
            fn(k)
        torch.cuda.synchronize()
        return (time.perf_counter() - t0) / n * 1e6

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
    for k in range(n):
        flush()
        evs[k][0].record(stream)
        replay(k)
        evs[k][1].record(stream)
    torch.cuda.synchronize()
    return {"step_ms": statistics.mean(a.elapsed_time(b) for a, b in evs),
            "wall_us_per_step_graph": wall(replay), "wall_us_per_step_eager": wall(eager),
            "note": "wall: steps issued back to back without L2 flush, synchronised once at the end; eager = "
                    "EngramLayer.decode (Python binding + C entry points per step)"}


def oracle_wkv(inp):
    """wkv as float64 for the oracle (made once per run)."""
    from workloads import bf16_bits_to_f64
    if "wkv_f64" not in inp:
        inp["wkv_f64"] = bf16_bits_to_f64(inp["lw"].wkv_bits)
    return inp["wkv_f64"]


def decode_cpu_baseline(w, inp, dw, n_steps):
    """The oracle on the first n_steps decode steps of the same 256 sequences.
    The carried histories come from the oracle's prefill of each prefix's last
    three tokens (a history is the last three compressed ids, so this equals
    the whole prefix's)."""
    from oracle import hashing as OH
    from oracle import layout as OL
    from oracle import pipeline as OP
    from workloads import bf16_bits_to_f64, residual_bits, table_rows

    tm = inp["tm"]
    lay_o = OL.build_layout(w.v, w.base_rows, [w.layer_id], pad_id=int(tm[0]))
    cu = dw.prefix.cu_seqlens
    tails = [dw.prefix.raw_ids[max(cu[s], cu[s + 1] - 3):cu[s + 1]] for s in range(len(cu) - 1)]
    tcu = np.concatenate([[0], np.cumsum([len(t) for t in tails])]).astype(np.int64)
    _, _, hist = OH.hash_prefill(np.concatenate(tails), tcu, tm, lay_o, 0)
    B = len(tails)
    slots = np.arange(B)
    W = oracle_wkv(inp)
    h = bf16_bits_to_f64(residual_bits(B, w.hc, w.hidden, w.seed))
    t0 = time.perf_counter()
    for k in range(n_steps):
        res = OP.layer_decode_step(lay_o, 0, dw.steps[k], slots, hist, tm, lambda r: table_rows(w.seed, r), W, h,
                                   inp["lw"].q_w, inp["lw"].k_w)
        hist, h = res.hist, res.h_out
    dt = time.perf_counter() - t0
    return {"value": B * n_steps / dt, "unit": "tokens/s", "steps_per_s": n_steps / dt, "cores": os.cpu_count(),
            "kind": "oracle", "sample": f"first {n_steps} decode steps of the {B} sequences, full layer per step "
                                        f"(numpy fp64, BLAS threads = all cores); {dt:.1f} s"}


def fp8_weights(w, inp, dev):
    """Block-FP8 wkv of the workload, packed for the projection (made once per run)."""
    if "fp8_wkv" not in inp:
        import torch
        import hashed_gram_conditional_gb300 as eg
        from workloads import mxfp8_weights

        K, N = 24 * 256, (w.hc + 1) * w.hidden
        w8, sf = mxfp8_weights(K, N, w.seed)
        inp["fp8_wkv"] = eg.engram_pack_wkv_fp8(torch.from_numpy(w8).to(dev), torch.from_numpy(sf).to(dev))
    return inp["fp8_wkv"]


def fp8_bench(args, w, inp, layer, flush, dev):
    """The layer with block-FP8 weights: the fused hash + gather copying the
    rows as stored (E4M3 + E8M0) and the block-scaled tensor-core projection
    with the gate and residual, on the same batch and table."""
    import torch
    import hashed_gram_conditional_gb300 as eg

    K, N = 24 * 256, (w.hc + 1) * w.hidden
    w8p, sfb = fp8_weights(w, inp, dev)
    b = inp["batch"]
    T = len(b.raw_ids)
    raw = torch.from_numpy(b.raw_ids).to(dev)
    cu = torch.from_numpy(b.cu_seqlens).to(dev)
    h = inp["bf16"](inp["h_bits"])
    hist = torch.full((w.n_seqs, 3), layer.layout.pad_id, dtype=torch.int32, device=dev)
    e8 = torch.empty((T, K), dtype=torch.uint8, device=dev)
    sfa = torch.empty((2 * 24, eg.sf_cols(T)), dtype=torch.int32, device=dev)
    mask = torch.empty(T, dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def run(ev=None):
        if ev is not None:
            ev[0].record(stream)
        eg.engram_hash_gather_fp8(layer.layout, 0, raw, cu, layer.token_map, layer.table, hist, e8, sfa, mask, None,
                                  status)
        if ev is not None:
            ev[1].record(stream)
        # the two kernels engram_project_gate_fp8 runs, with an event between them
        eg.engram_project_fp8(e8, sfa, w8p, sfb, h, layer.q_w, layer.k_w, bufs["partials"], bufs["v"], status)
        if ev is not None:
            ev[3].record(stream)
        eg.engram_gate_add(bufs["partials"], bufs["v"], h, mask, layer.eps, layer.clamp, layer.score_scale)
        if ev is not None:
            ev[2].record(stream)

    bufs = layer._buffers(T, dev)
    for _ in range(5):
        flush()
        run()
    n = args.fp8_steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n)]
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for k in range(n):
        flush()
        run(evs[k])
    torch.cuda.synchronize()
    timed = time.perf_counter() - t0
    step = statistics.mean(ev[0].elapsed_time(ev[2]) for ev in evs) / 1e3
    pg = statistics.mean(ev[1].elapsed_time(ev[2]) for ev in evs) / 1e3
    proj = statistics.mean(ev[1].elapsed_time(ev[3]) for ev in evs) / 1e3
    hg = statistics.mean(ev[0].elapsed_time(ev[1]) for ev in evs) / 1e3
    flops = 2.0 * T * K * N
    out = {}
    if not args.no_cpu_baseline:
        from oracle import dequant as OD
        from oracle import pipeline as OP
        from workloads import bf16_bits_to_f64, mxfp8_weights
        n_o, raw_o, cu_o, tm_o, lay_o, table_o = oracle_prefix(w, inp, 2048)
        W8 = OD.dequant_mx_weights(*mxfp8_weights(K, N, w.seed))
        h_o = bf16_bits_to_f64(inp["h_bits"][:n_o])
        out["cpu_baseline"] = oracle_timed(
            lambda: OP.layer_forward(lay_o, 0, raw_o, cu_o, tm_o, table_o, W8, h_o, inp["lw"].q_w, inp["lw"].k_w),
            n_o, f"first {n_o} packed positions, one full layer pass with the dequantised block-FP8 wkv")
        del W8
    return {**out, "workload": f"{w.name} batch ({T} tokens), block-FP8 wkv (E4M3, E8M0 per 32 of k), L2 flushed",
            "steps": n, "step_ms": step * 1e3, "tokens_per_s": T / step, "hash_gather_ms": hg * 1e3,
            "project_gate_ms": pg * 1e3, "project_ms": proj * 1e3, "gate_ms": (pg - proj) * 1e3,
            "project_tflops": flops / proj / 1e12, "timed_s": timed,
            "kernels": "gather_ldgsts_kernel<HashedRows, Fp8Out>, project8_kernel<unfused>, gate_add_kernel "
                       "(what engram_hash_gather_fp8 + engram_project_gate_fp8 run)",
            "hash_gather_bytes_per_token": 4 + 24 * 264 + 24 * 256 + 24 * 8,
            "device_status": int(status.item())}


def generic_bench(args, w, flush, dev):
    """The Engram-27B shape of the Engram paper on the same token batch shape:
    2/3-grams x 8 heads = 16 columns of plain bf16 rows of 80 elements
    (K = 1280), hidden 2560, 4 streams, table from base 2,000,000 (~32 M rows,
    5.1 GB), filled on the device."""
    import torch
    import hashed_gram_conditional_gb300 as eg
    from workloads import Workload, layer_weights, prefill_batch, residual_bits, token_map

    R = 80
    wg = Workload("generic27b", w.v_raw, w.v, w.base_rows, 15, w.n_seqs, w.seq_len, 2560, 4, w.dead_frac,
                  seed=w.seed)
    tm = token_map(wg.v_raw, wg.v, wg.seed)
    lay = eg.build_layout(wg.v, wg.base_rows, [2, 15], max_ngram=3, n_heads=8, pad_id=int(tm[0]),
                          expected_vocab=wg.v)
    total = lay.total_rows(1)
    table = eg.engram_fill_synthetic_rows_bf16(torch.empty((total, R), dtype=torch.bfloat16, device=dev), wg.seed)
    lw = layer_weights(wg, n_cols=lay.n_cols, row_dim=R)

    def bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

    layer = eg.EngramLayer(lay, 1, table, torch.from_numpy(tm).to(dev), eg.engram_pack_wkv(bf16(lw.wkv_bits)),
                           torch.from_numpy(lw.q_w).to(dev), torch.from_numpy(lw.k_w).to(dev))
    b = prefill_batch(wg, seed=wg.seed)
    T = len(b.raw_ids)
    raw = torch.from_numpy(b.raw_ids).to(dev)
    cu = torch.from_numpy(b.cu_seqlens).to(dev)
    h = bf16(residual_bits(T, wg.hc, wg.hidden, wg.seed))
    hist = torch.full((wg.n_seqs, 2), lay.pad_id, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    bufs = layer._buffers(T, dev)
    stream = torch.cuda.current_stream(dev)

    def run(ev=None):
        if ev is not None:
            ev[0].record(stream)
        eg.engram_hash_gather_rows_bf16(lay, 1, raw, cu, layer.token_map, table, hist, bufs["e"], bufs["mask"], None,
                                        status)
        if ev is not None:
            ev[1].record(stream)
        # the two kernels engram_project_gate runs at K < 3200, with an event between them
        eg.engram_project(bufs["e"], layer.wkv_packed, h, layer.q_w, layer.k_w, bufs["partials"], bufs["v"], status)
        if ev is not None:
            ev[3].record(stream)
        eg.engram_gate_add(bufs["partials"], bufs["v"], h, bufs["mask"], layer.eps, layer.clamp, layer.score_scale)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(3):
        flush()
        run()
    n = args.generic_steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n)]
    for k in range(n):
        flush()
        run(evs[k])
    torch.cuda.synchronize()
    step = statistics.mean(ev[0].elapsed_time(ev[2]) for ev in evs) / 1e3
    hg = statistics.mean(ev[0].elapsed_time(ev[1]) for ev in evs) / 1e3
    proj = statistics.mean(ev[1].elapsed_time(ev[2]) for ev in evs) / 1e3
    proj_only = statistics.mean(ev[1].elapsed_time(ev[3]) for ev in evs) / 1e3
    gate_only = statistics.mean(ev[3].elapsed_time(ev[2]) for ev in evs) / 1e3
    C = lay.n_cols
    hg_bytes = 4 + 2 * C * R * 2
    flops = 2.0 * C * R * (wg.hc + 1) * wg.hidden
    base = {}
    if not args.no_cpu_baseline:
        from oracle import dequant as OD
        from oracle import layout as OL
        from oracle import pipeline as OP
        from workloads import bf16_bits_to_f64, table_rows_bf16
        n_o = 2048
        cu_o = np.minimum(b.cu_seqlens, n_o)
        cu_o = cu_o[: int(np.searchsorted(cu_o, n_o)) + 1]
        lay_o = OL.build_layout(wg.v, wg.base_rows, [2, 15], max_ngram=3, n_heads=8, pad_id=int(tm[0]))
        W = bf16_bits_to_f64(lw.wkv_bits)
        h_o = bf16_bits_to_f64(residual_bits(n_o, wg.hc, wg.hidden, wg.seed))
        base["cpu_baseline"] = oracle_timed(
            lambda: OP.layer_forward(lay_o, 1, b.raw_ids[:n_o], cu_o, tm,
                                     lambda r: bf16_bits_to_f64(table_rows_bf16(wg.seed, r, R)), W, h_o, lw.q_w,
                                     lw.k_w, gather=OD.gather_rows),
            n_o, f"first {n_o} packed positions, one full layer pass")
    out = {"workload": f"{T} tokens ({wg.n_seqs} x {wg.seq_len}), 2/3-grams x 8 heads = {C} rows of {R} bf16, "
                       f"table {total} rows ({total * R * 2 / 1e9:.1f} GB), hidden {wg.hidden}, hc {wg.hc}, "
                       "L2 flushed", "steps": n,
           "step_ms": step * 1e3, "tokens_per_s": T / step, "hash_gather_ms": hg * 1e3,
           "hash_gather_gbs": hg_bytes * T / hg / 1e9, "hash_gather_bytes_per_token": hg_bytes,
           "project_gate_ms": proj * 1e3, "project_gate_tflops": flops * T / proj / 1e12,
           "project_ms": proj_only * 1e3, "project_tflops": flops * T / proj_only / 1e12,
           "gate_ms": gate_only * 1e3,
           "gate_gbs": GATE_BYTES_PER_TOKEN(wg.hc, wg.hidden) * T / gate_only / 1e9,
           "device_status": int(status.item()), **base}
    del table
    return out


def conv_bench(args, w, inp, layer, flush, dev):
    """The original Engram layer (short convolution, kernel 4, dilation 3) on the
    same batch: hash -> gather -> projection -> gates -> convolution + residual."""
    import torch
    import hashed_gram_conditional_gb300 as eg
    from workloads import conv_weights

    cw, gamma = conv_weights(4, w.hc, w.hidden, w.seed)
    cl = eg.EngramLayer(layer.layout, layer.layer, layer.table, layer.token_map, layer.wkv_packed, layer.q_w,
                        layer.k_w, conv=eg.ShortConv(torch.from_numpy(cw).to(dev), torch.from_numpy(gamma).to(dev), 3))
    b = inp["batch"]
    T = len(b.raw_ids)
    raw = torch.from_numpy(b.raw_ids).to(dev)
    cu = torch.from_numpy(b.cu_seqlens).to(dev)
    h = inp["bf16"](inp["h_bits"])
    ring, head = cl.new_conv_state(w.n_seqs, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    bufs = cl._buffers(T, dev)

    def run(ev=None):
        if ev is not None:
            ev[0].record(stream)
        eg.engram_hash(cl.layout, 0, raw, cu, cl.token_map, None, bufs["rows"], bufs["mask"], status)
        eg.engram_gather_dequant(cl.table, cl.total_rows, bufs["rows"], bufs["e"], status)
        eg.engram_project(bufs["e"], cl.wkv_packed, h, cl.q_w, cl.k_w, bufs["partials"], bufs["v"], status)
        g = eg.engram_gates(bufs["partials"], T, cl.hidden, cl.hc, bufs["mask"], cl.eps, cl.clamp, cl.score_scale,
                            bufs["gate"])
        if ev is not None:
            ev[1].record(stream)
        eg.engram_short_conv_add(g, bufs["v"], h, bufs["mask"], cl.conv.w, cl.conv.gamma, 3, cl.conv.eps, cu, None,
                                 ring, head, bufs["conv_ws"], status)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(3):
        flush()
        run()
    n = args.conv_steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
    for k in range(n):
        flush()
        run(evs[k])
    torch.cuda.synchronize()
    step = statistics.mean(ev[0].elapsed_time(ev[2]) for ev in evs) / 1e3
    conv_s = statistics.mean(ev[1].elapsed_time(ev[2]) for ev in evs) / 1e3
    cbytes = CONV_BYTES_PER_TOKEN(w.hc, w.hidden) * T
    out = {}
    if not args.no_cpu_baseline:
        from oracle import pipeline as OP
        from workloads import bf16_bits_to_f64
        n_o, raw_o, cu_o, tm_o, lay_o, table_o = oracle_prefix(w, inp, 2048)
        h_o = bf16_bits_to_f64(inp["h_bits"][:n_o])
        cp = OP.ConvParams(cw.astype(np.float64), gamma.astype(np.float64), 3)
        out["cpu_baseline"] = oracle_timed(
            lambda: OP.layer_forward_conv(lay_o, 0, raw_o, cu_o, tm_o, table_o, oracle_wkv(inp), h_o,
                                          inp["lw"].q_w, inp["lw"].k_w, cp),
            n_o, f"first {n_o} packed positions, one full layer pass with the short convolution")
    return {**out, "workload": f"{w.name} batch, kernel 4, dilation 3, state ring kept per sequence", "steps": n,
            "step_ms": step * 1e3, "tokens_per_s": T / step, "conv_ms": conv_s * 1e3,
            "conv_gbs": cbytes / conv_s / 1e9, "algorithmic_bytes": cbytes, "device_status": int(status.item()),
            "kernels": "conv_prep_kernel + conv_add_kernel + conv_state_kernel",
            "note": "projection + gates run as two kernels here (engram_project, gates-only engram_gate_add)"}


def host_table_bench(args, w, inp, layer, flush, dev, device_step_ms):
    """The same table in pinned host memory (Grace LPDDR).

    (a) zero-copy: the gather kernel reads the rows over NVLink-C2C;
    (b) prefetch (``EngramLayer.prefetch``): the hash on the compute stream,
        then on a copy stream the row ids go to the host, host threads copy the
        rows into pinned staging, one DMA moves them to HBM and they are
        dequantised; timed alone, then double-buffered so that fetching batch
        k+1 runs while batch k is projected.
    Four batches of the workload's shape (different seeds) rotate, so the rows
    gathered by the host do not stay in its caches from one step to the next.
    """
    import torch
    import hashed_gram_conditional_gb300 as eg
    from workloads import prefill_batch

    total = layer.total_rows
    t0 = time.perf_counter()
    try:
        host = torch.empty(total * eg.ROW_BYTES, dtype=torch.uint8, pin_memory=True)
    except RuntimeError as ex:
        return {"skipped": f"pinned host table of {total * eg.ROW_BYTES / 1e9:.2f} GB unavailable: {ex}"}
    pin_s = time.perf_counter() - t0
    eg.engram_fill_synthetic_table(host, total, w.seed, dev)
    torch.cuda.synchronize()
    hl = eg.EngramLayer(layer.layout, layer.layer, host, layer.token_map, layer.wkv_packed, layer.q_w, layer.k_w)
    n = args.host_steps
    batches = [prefill_batch(w, seed=w.seed + 1000 + i) for i in range(4)]
    T = len(batches[0].raw_ids)
    raws = [torch.from_numpy(b.raw_ids).to(dev) for b in batches]
    cus = [torch.from_numpy(b.cu_seqlens).to(dev) for b in batches]
    C = layer.layout.n_cols
    rows = torch.empty((T, C), dtype=torch.int32, device=dev)
    e = torch.empty((T, C * 256), dtype=torch.bfloat16, device=dev)
    h = inp["bf16"](inp["h_bits"][:T])
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    main = torch.cuda.current_stream(dev)
    side = torch.cuda.Stream(dev)
    row_bytes = T * C * eg.ROW_BYTES
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]

    # (a) zero-copy gather over NVLink-C2C
    zc = []
    for k in range(n + 3):
        eg.engram_hash(layer.layout, 0, raws[k % 4], cus[k % 4], layer.token_map, None, rows, None)
        flush()
        ev[0].record(main)
        eg.engram_gather_dequant(host, total, rows, e, status)
        ev[1].record(main)
        ev[1].synchronize()
        if k >= 3:
            zc.append(ev[0].elapsed_time(ev[1]))

    # (b1) the prefetch alone: from the hash to the rows being ready
    fe, bad = [], 0
    for k in range(n + 3):
        ev[0].record(main)
        pf = hl.prefetch(raws[k % 4], cus[k % 4], status=status, copy_stream=side)
        main.wait_event(pf.ready)
        ev[1].record(main)
        ev[1].synchronize()
        bad += pf.bad_rows
        hl.prefill_prefetched(pf, h, status)
        if k >= 3:
            fe.append(ev[0].elapsed_time(ev[1]))
    torch.cuda.synchronize()

    # (b2) double-buffered: the fetch of batch k+1 overlaps the projection of batch k
    def pipeline(steps):
        pf = hl.prefetch(raws[0], cus[0], status=status, copy_stream=side)
        for k in range(steps):
            nxt = hl.prefetch(raws[(k + 1) % 4], cus[(k + 1) % 4], status=status, copy_stream=side) \
                if k + 1 < steps else None
            hl.prefill_prefetched(pf, h, status)
            pf = nxt

    pipeline(3)
    flush()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    ev[0].record(main)
    pipeline(n)
    ev[1].record(main)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    pipe_ms = ev[0].elapsed_time(ev[1]) / n
    zc_ms, fetch_ms = statistics.mean(zc), statistics.mean(fe)
    return {"workload": f"{w.name}: 4 rotating batches of {T} tokens, {total * eg.ROW_BYTES / 1e9:.2f} GB table "
                        "in pinned host memory", "steps": n, "pin_alloc_s": pin_s,
            "zero_copy_gather_ms": zc_ms, "zero_copy_row_gbs": row_bytes / zc_ms / 1e6,
            "prefetch_ms": fetch_ms, "prefetch_row_gbs": row_bytes / fetch_ms / 1e6,
            "pipelined_step_ms": pipe_ms, "pipelined_tokens_per_s": T / pipe_ms * 1e3,
            "pipelined_wall_tokens_per_s": T * n / wall,
            "device_table_step_ms": device_step_ms,
            "host_threads": int(os.environ.get("OMP_NUM_THREADS", "0")) or os.cpu_count(),
            "bad_rows": bad, "device_status": int(status.item()), "row_bytes_per_step": row_bytes,
            "note": "L2 flushed before each zero-copy gather; the pipelined steps run back to back"}


# ------------------------------------------------------------------------- oracle timing


def oracle_sample(w, inp, n_tokens):
    """Prepare a bounded oracle run over the first n_tokens packed positions of the batch."""
    from oracle import hashing as OH
    from oracle import layout as OL
    from oracle import pipeline as OP
    from workloads import bf16_bits_to_f64, table_rows

    b = inp["batch"]
    n = min(n_tokens, len(b.raw_ids))
    raw = b.raw_ids[:n]
    cu = np.minimum(b.cu_seqlens, n)
    cu = cu[: int(np.searchsorted(cu, n)) + 1]
    tm = inp["tm"]
    lay_o = OL.build_layout(w.v, w.base_rows, [w.layer_id], pad_id=int(tm[0]))
    rows, _, _ = OH.hash_prefill(raw, cu, tm, lay_o, 0)
    uniq = np.unique(rows)
    cache = dict(zip(uniq.tolist(), table_rows(w.seed, uniq)))   # table bytes, read by the oracle below

    def table(r):
        return np.stack([cache[int(x)] for x in r])

    W = oracle_wkv(inp)
    h = bf16_bits_to_f64(inp["h_bits"][:n])

    def run():
        return OP.layer_forward(lay_o, 0, raw, cu, tm, table, W, h, inp["lw"].q_w, inp["lw"].k_w)
    return n, run


def oracle_timed(run, n, label):
    """Time one bounded oracle run (the oracle as it stands) as a cpu_baseline entry."""
    t0 = time.perf_counter()
    run()
    dt = time.perf_counter() - t0
    return {"value": n / dt, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{label} (numpy fp64, BLAS threads = all cores); {dt:.1f} s"}


def oracle_prefix(w, inp, n_tokens):
    """The first n_tokens packed positions of the batch, their layout and table reader for the oracle."""
    from oracle import hashing as OH
    from oracle import layout as OL
    from workloads import table_rows

    b = inp["batch"]
    n = min(n_tokens, len(b.raw_ids))
    raw = b.raw_ids[:n]
    cu = np.minimum(b.cu_seqlens, n)
    cu = cu[: int(np.searchsorted(cu, n)) + 1]
    tm = inp["tm"]
    lay_o = OL.build_layout(w.v, w.base_rows, [w.layer_id], pad_id=int(tm[0]))
    rows, _, _ = OH.hash_prefill(raw, cu, tm, lay_o, 0)
    uniq = np.unique(rows)
    cache = dict(zip(uniq.tolist(), table_rows(w.seed, uniq)))   # table bytes, read by the oracle below

    def table(r):
        return np.stack([cache[int(x)] for x in r])
    return n, raw, cu, tm, lay_o, table


def cpu_baseline(w, inp, n_tokens):
    n, run = oracle_sample(w, inp, n_tokens)
    t0 = time.perf_counter()
    run()
    dt = time.perf_counter() - t0
    return {"value": n / dt, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"first {n} packed positions of the same batch, one full layer pass "
                      f"(numpy fp64, BLAS threads = all cores); {dt:.1f} s"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    from workloads import WORKLOADS
    w = WORKLOADS[args.workload]
    # inputs are generated on the host; no GPU work on this arm
    from workloads import layer_weights, prefill_batch, residual_bits, token_map
    tm = token_map(w.v_raw, w.v, w.seed)
    b = prefill_batch(w, seed=w.seed)
    inp = dict(tm=tm, lw=layer_weights(w), batch=b, h_bits=residual_bits(len(b.raw_ids), w.hc, w.hidden, w.seed))
    n, run = oracle_sample(w, inp, args.ref_sample)
    for _ in range(args.warmup):
        run()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        run()
        times.append(time.perf_counter() - t0)
    tot = sum(times)
    value = n * args.steps / tot
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": tot / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (same seeded inputs as the GPU arm)",
        "config": {"workload": workload_desc(w), "tokens_per_step": n,
                   "note": "each step is the CPU oracle on a bounded sample of the workload"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                         "sample": f"first {n} packed positions of the batch per step"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        out = run_reference(args, rank, world)
    else:
        import torch
        if world > 1:
            import torch.distributed as dist
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            dist.init_process_group(backend="nccl", device_id=torch.device("cuda", local))
        out = run_ours(args, rank, world, local)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
