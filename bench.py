#!/usr/bin/env python3
"""Benchmark of the skinny Q4K x bf16 product on GB300: weight-read GB/s, % of the HBM
roofline and ms per 15.8 GB weight pass, per M.

Workload of a step (default): one full 64-layer weight pass of the 27B hybrid model's Q4K
matrices (per layer q 5120x5120, k and v 1024x5120, o 5120x5120, gate_up 34816x5120,
down 5120x17408: 384 matrices, 11.89 GB of packed weights) through ONE qmm_run_batched call
with M activation rows (M = 8 by default: the pages' 8-row verify pass).  The weights are far
larger than L2 (129 MB), so no flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--M 8] [--impl ours|reference]
  python bench.py --single gate_up|down|q|k|lm_head|all [--Ms 1,2,...] [--variant fma|tc|auto|both]
  python bench.py --ffn [--Ms 1,2,...]     (one feed-forward block per call: gate/up, gate, down)
  python bench.py --indexed [--Ms 1,2,...] (indexed-expert product over 16 experts)
  python bench.py --profile-pass L [--M 8] (a few untimed steps over the first L layers: the small
                                           case that DRAM-traffic captures run on)

`--single` times one matrix product per launch instead (weights cycled over copies totalling
more than 4x the L2 size), for the switch-point sweep between the two kernel families and as
the small case that profiling runs on.

Under torchrun each rank runs its own full pass on its own GPU (independent problems, no
collective on the data path); the timing is the max over ranks and `value` sums all ranks'
weight bytes.  `--impl reference` times the oracle (plain fp64 C on the host cores) on a
bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "weight-read GB/s and % of HBM roofline vs M (1..32); ms per 15.8 GB pass"
UNIT = "GB/s"
PASS_BYTES = 15.8e9          # the pages' weight pass ("sixi-asi 0.9", section "The patch")
SPEC_HBM_GBS = 8000.0        # GB300 HBM3e, nominal
LAYERS = 64


# ----------------------------------------------------------------------------- metric ----

def weight_gbps(weight_bytes: float, ms: float) -> float:
    """Weight-only effective bandwidth: packed weight bytes read / kernel time (GB/s)."""
    return weight_bytes / (ms * 1e-3) / 1e9


def ms_per_pass(gbps: float) -> float:
    return PASS_BYTES / (gbps * 1e9) * 1e3


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            return json.load(fh)
    except OSError:
        return None


def hbm_peak():
    mp = measured_peaks()
    if mp and mp.get("hbm_gbs"):
        return float(mp["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_source_hash() -> str:
    """Hash of the library's sources with // comments and blank space removed (a comment edit
    does not change the kernels whose counters a profile recorded)."""
    import re
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "bit_quantized_skinny_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), encoding="utf-8") as fh:
            code = re.sub(r"//[^\n]*", "", fh.read())
        h.update(name.encode() + " ".join(code.split()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str, M: int):
    """DRAM bytes of one step (all its product launches) from a committed ncu summary, if taken on
    the current sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as fh:
            rec = json.load(fh)
    except (OSError, ValueError):
        return None
    key = f"{kernel}|{workload}|M={M}"
    ent = rec.get(key)
    if not ent or ent.get("source_hash") != kernel_source_hash():
        return None
    return ent.get("dram_bytes_per_step")


# ----------------------------------------------------------------------------- clocks ----

class ClockSampler:
    """Samples SM clock and clock-event reasons through NVML (ctypes) during a region."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown", 0x2: "applications_clocks"}

    def __init__(self, cuda_device: int, interval_s: float = 0.002):
        self.ok = False
        self.samples = []
        self.interval = interval_s
        self._stop = threading.Event()
        try:
            import torch
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                return
            self.handle = ctypes.c_void_p()
            uuid = str(torch.cuda.get_device_properties(cuda_device).uuid)
            uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            if self.nvml.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.handle)) != 0:
                return
            mx = ctypes.c_uint(0)
            self.nvml.nvmlDeviceGetMaxClockInfo(self.handle, 1, ctypes.byref(mx))
            self.max_mhz = mx.value
            self._reason_fn = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                self.nvml.nvmlDeviceGetCurrentClocksThrottleReasons
            self.ok = True
        except Exception:
            self.ok = False

    def _poll(self):
        clk = ctypes.c_uint(0)
        rs = ctypes.c_ulonglong(0)
        while not self._stop.is_set():
            if self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(clk)) == 0 and \
                    self._reason_fn(self.handle, ctypes.byref(rs)) == 0:
                self.samples.append((clk.value, rs.value))
            time.sleep(self.interval)

    def __enter__(self):
        if self.ok:
            self._t = threading.Thread(target=self._poll, daemon=True)
            self._t.start()
        return self

    def __exit__(self, *exc):
        if self.ok:
            self._stop.set()
            self._t.join()

    def summary(self):
        if not self.ok or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": getattr(self, "max_mhz", None), "reasons": [],
                    "samples": 0, "source": "nvml unavailable" if not self.ok else "no samples"}
        reasons = set()
        for _, r in self.samples:
            for bit, name in self.REASONS.items():
                if r & bit:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(c for c, _ in self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(reasons), "samples": len(self.samples), "source": "nvml"}


# ----------------------------------------------------------------------------- workload --

def layer_pass_setup(M: int, device: str, layers: int = LAYERS):
    """Device buffers for the 64-layer pass (or its first `layers` layers): each distinct matrix
    is packed once and copied into one distinct device buffer per layer (content does not change
    the speed; every buffer is read from HBM).  Returns (entries, info) with info holding the
    host-side copies."""
    import torch
    from bit_quantized_skinny_gb300 import inputs, qmm, workloads

    bases, hosts = [], []
    for idx, (name, N, K) in enumerate(workloads.LAYER_SHAPES):
        Wd, Wh = workloads.packed_weights(N, K, inputs.seed_for(4, idx), device=device, keep_host=True)
        bases.append(Wd)
        hosts.append(Wh)
    xs = {}
    for K in sorted({K for _, _, K in workloads.LAYER_SHAPES}):
        xs[K] = workloads.activations(M, K, inputs.seed_for(4, 100 + K % 97), device=device)
    # the outputs of a pass live in one arena (one result buffer per step, as a model runtime
    # keeps them), each product's Y a slice of it
    y_arena = torch.empty(layers * sum(M * N for _, N, _ in workloads.LAYER_SHAPES), dtype=torch.float32,
                          device=device)
    items, ys, ws = [], [], []
    off = 0
    for layer in range(layers):
        for idx, (name, N, K) in enumerate(workloads.LAYER_SHAPES):
            w = bases[idx] if layer == 0 else bases[idx].clone()
            y = y_arena[off:off + M * N].view(M, N)
            off += M * N
            ws.append(w)
            ys.append(y)
            items.append((w, xs[K][0], y, N, K))
    entries = qmm.make_entries(items)
    weight_bytes = sum(w.numel() for w in ws)
    algo_bytes = weight_bytes + sum(M * K * 2 + M * N * 4 for _, _, _, N, K in items)
    return entries, dict(items=items, ws=ws, ys=ys, y_arena=y_arena, xs=xs, hosts=hosts,
                         weight_bytes=weight_bytes, algo_bytes=algo_bytes)


def aggregate_ranks(ms: float, weight_bytes: int, dist_ok: bool, device=None):
    """The step time of the job (the max over ranks) and the weight bytes all ranks streamed per
    step (every rank runs its own full pass on its own GPU: weak scaling, no collective on the
    data path; this is the only exchange, after the timed region)."""
    if not dist_ok:
        return ms, weight_bytes
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64)
    b = torch.tensor([float(weight_bytes)], dtype=torch.float64)
    if device is not None:
        t, b = t.to(device), b.to(device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(b, op=dist.ReduceOp.SUM)
    return float(t.item()), int(b.item())


def time_steps(fn, steps: int, warmup: int, stream, sync_ranks):
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    sync_ranks()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    sync_ranks()
    return e0.elapsed_time(e1) / steps


def time_trials(fn, steps: int, warmup: int, stream, sync_ranks, trials: int = 5):
    """`trials` timed regions of exactly `steps` steps each (the warm-up before the first):
    the per-step times of the trials."""
    out = [time_steps(fn, steps, warmup, stream, sync_ranks)]
    for _ in range(trials - 1):
        out.append(time_steps(fn, steps, 0, stream, sync_ranks))
    return out


class RooflineGuard:
    """A result that implies reading HBM faster than the memory system can is a bug ("sixi-asi
    0.9", section "The patch": a pass faster than the bandwidth floor was a bug, not a win).  The
    ceiling is the read-only probe of this run (qmm_stream_read), 3 % slack; before it is measured,
    the measured copy bandwidth plus 15 % (a read-only stream can beat a copy), else the
    8 TB/s spec."""

    def __init__(self):
        self.read_gbps = None

    def ceiling(self):
        if self.read_gbps:
            return 1.03 * self.read_gbps
        mp = measured_peaks()
        if mp and mp.get("hbm_gbs"):
            return 1.15 * float(mp["hbm_gbs"])
        return SPEC_HBM_GBS

    def check(self, gbps: float, where: str):
        if gbps > self.ceiling():
            raise SystemExit(f"roofline guard: {where}: {gbps:.0f} GB/s exceeds the {self.ceiling():.0f} GB/s "
                             f"ceiling; a benchmark that beats the roofline is a bug report")
        return gbps


GUARD = RooflineGuard()


def peak_probes(device: str):
    """HBM peak probes on this GPU (FlashRT issue #153: the device-to-device bandwidth check and the
    sustained-read microtest): the read-only streaming kernel qmm_stream_read over a 4 GiB buffer
    (burst: one pass, median of 5; sustained: back-to-back passes for about 100 ms) and a 1 GiB
    device-to-device copy (read + write bytes, median of 5)."""
    import torch
    from bit_quantized_skinny_gb300 import qmm

    stream = torch.cuda.current_stream()
    nbytes = 4 << 30
    buf = torch.ones(nbytes // 4, dtype=torch.int32, device=device)
    sink = torch.empty(qmm.stream_read_sink_words(), dtype=torch.int32, device=device)
    rd = lambda: qmm.stream_read(buf, sink)
    burst = statistics.median(time_trials(rd, 1, 3, stream, lambda: None, trials=5))
    passes = max(3, int(100.0 / burst))
    sustained = time_steps(rd, passes, 1, stream, lambda: None)
    src = torch.empty(1 << 30, dtype=torch.uint8, device=device)
    dst = torch.empty_like(src)
    cp = lambda: dst.copy_(src)
    copy_ms = statistics.median(time_trials(cp, 1, 3, stream, lambda: None, trials=5))
    del buf, sink, src, dst
    torch.cuda.empty_cache()
    out = {"read_burst_gbps": round(weight_gbps(nbytes, burst), 1),
           "read_sustained_gbps": round(weight_gbps(nbytes, sustained), 1),
           "read_sustained_ms": round(passes * sustained, 1),
           "d2d_copy_gbps_read_plus_write": round(weight_gbps(2 << 30, copy_ms), 1),
           "d2d_copy_payload_gbps": round(weight_gbps(1 << 30, copy_ms), 1),
           "how": "qmm_stream_read (this library's read-only streaming kernel) over 4 GiB; torch copy_ of 1 GiB"}
    GUARD.read_gbps = max(out["read_burst_gbps"], out["read_sustained_gbps"])
    return out


def graph_launch_us(fns, stream, trials: int = 5, min_launches: int = 20):
    """Device time per launch under CUDA-graph replay: the launches (one per weight copy, the list
    repeated to at least min_launches) captured once into a graph on a side stream (after one
    eager pass there, which sizes the tensor-core workspace), replayed once, then CUDA events on
    the launching stream around `reps` replays per trial; the median over the trials, in us."""
    import torch
    seq = list(fns)
    while len(seq) < min_launches:
        seq += list(fns)
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for f in fns:
            f()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            for f in seq:
                f()
    stream.wait_stream(side)
    graph.replay()
    torch.cuda.synchronize()
    reps = 3
    times = []
    for _ in range(trials):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            graph.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) / (reps * len(seq)))
    del graph
    return statistics.median(times) * 1e3


SWITCH_MS = [1, 2, 3, 4, 7, 8, 9, 12, 16]


def config_timings(device: str):
    """The configurations other than the pass, device-timed under CUDA-graph replay, weights
    cycled over copies totalling at least 4x L2 (each launch reads HBM):
      ffn_decode_m1  single FFN layer at M = 1: the gate/up product 34816 x 5120, the down product
                     5120 x 17408, and the block (qmm_run_ffn, qmm_run_ffn_fused)
      lm_head        N = 248320, K = 5120 at M = 1 and M = 7
      switch_point   gate_up, down, q (5120 x 5120), k (1024 x 5120) at M in SWITCH_MS, both kernel
                     families, and the family the dispatcher picks
    Each figure: us per launch, GB/s of packed weights, fraction of the read probe."""
    import torch
    from bit_quantized_skinny_gb300 import inputs, qmm, workloads

    stream = torch.cuda.current_stream()
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    peak = GUARD.read_gbps or hbm_peak()[0]

    def weights(N, K, seed, min_bytes=4 * l2):
        w = workloads.packed_weights_fmt(qmm.FMT_Q4K, N, K, seed)
        return [w] + [w.clone() for _ in range(max(1, -(-min_bytes // w.numel())) - 1)]

    def fig(us, wbytes, where):
        g = GUARD.check(weight_gbps(wbytes, us * 1e-3), where)
        return {"us": round(us, 2), "gbps": round(g, 1), "frac_of_read_peak": round(g / peak, 4)}

    out = {}
    # FFN layer decode, M = 1
    F, K = 17408, 5120
    gu = weights(2 * F, K, inputs.seed_for(2, 0))
    dn = weights(K, F, inputs.seed_for(2, 1))
    M = 1
    X, _ = workloads.activations(M, K, inputs.seed_for(2, 51), device=device)
    Xd, _ = workloads.activations(M, F, inputs.seed_for(2, 52), device=device)
    Yg = torch.empty((M, 2 * F), device=device)
    Yd = torch.empty((M, K), device=device)
    ffn = {"gate_up": fig(graph_launch_us([lambda w=w: qmm.run(w, 2 * F, K, X, Yg, M=M) for w in gu], stream),
                          gu[0].numel(), "ffn gate_up M=1"),
           "down": fig(graph_launch_us([lambda w=w: qmm.run(w, K, F, Xd, Yd, M=M) for w in dn], stream),
                       dn[0].numel(), "ffn down M=1")}
    ffn["gate_up"]["variant"] = qmm.VARIANT_NAMES[qmm.select_variant(M, 2 * F, K)]
    ffn["down"]["variant"] = qmm.VARIANT_NAMES[qmm.select_variant(M, K, F)]
    ws = torch.empty(qmm.ffn_workspace_bytes(M, F), dtype=torch.uint8, device=device)
    wsf = torch.empty(qmm.ffn_fused_workspace_bytes(M, F), dtype=torch.uint8, device=device)
    pairs = list(zip(gu, dn))[:max(4, -(-4 * l2 // (gu[0].numel() + dn[0].numel())))]
    blk = gu[0].numel() + dn[0].numel()
    ffn["block"] = fig(graph_launch_us([lambda g=g, d=d: qmm.run_ffn(g, d, F, K, X, Yd, ws, M=M) for g, d in pairs],
                                       stream), blk, "ffn block M=1")
    ffn["block_fused"] = fig(graph_launch_us([lambda g=g, d=d: qmm.run_ffn_fused(g, d, F, K, X, Yd, wsf, M=M)
                                              for g, d in pairs], stream), blk, "ffn fused block M=1")
    out["ffn_decode_m1"] = ffn
    # the switch-point table (gate_up and down reuse the copies above)
    qw = weights(5120, 5120, inputs.seed_for(3, 2))
    kw = weights(1024, 5120, inputs.seed_for(3, 3))
    table = {}
    for name, ws_, N, Kk in (("gate_up", gu, 2 * F, K), ("down", dn, K, F), ("q", qw, 5120, 5120), ("k", kw, 1024, 5120)):
        rows = {}
        for m in SWITCH_MS:
            Xm, _ = workloads.activations(m, Kk, inputs.seed_for(3, 60 + m), device=device)
            Ym = torch.empty((m, N), device=device)
            row = {"picks": qmm.VARIANT_NAMES[qmm.select_variant(m, N, Kk)]}
            for v in (qmm.VARIANT_FMA, qmm.VARIANT_TC):
                us = graph_launch_us([lambda w=w, v=v: qmm.run(w, N, Kk, Xm, Ym, M=m, variant=v) for w in ws_], stream)
                f = fig(us, ws_[0].numel(), f"switch {name} M={m} {qmm.VARIANT_NAMES[v]}")
                row[qmm.VARIANT_NAMES[v]] = {"us": f["us"], "gbps": f["gbps"]}
            rows[str(m)] = row
        table[name] = {"N": N, "K": Kk, "weight_bytes": ws_[0].numel(), "copies": len(ws_), "per_M": rows}
    out["switch_point"] = table
    del gu, dn, qw, kw, pairs
    torch.cuda.empty_cache()
    # lm_head
    N, K = 248320, 5120
    lw = weights(N, K, inputs.seed_for(5, 0))
    lm = {}
    for m in (1, 7):
        Xm, _ = workloads.activations(m, K, inputs.seed_for(5, 70 + m), device=device)
        Ym = torch.empty((m, N), device=device)
        f = fig(graph_launch_us([lambda w=w: qmm.run(w, N, K, Xm, Ym, M=m) for w in lw], stream), lw[0].numel(),
                f"lm_head M={m}")
        f["variant"] = qmm.VARIANT_NAMES[qmm.select_variant(m, N, K)]
        lm[f"M{m}"] = f
    out["lm_head"] = lm
    del lw
    torch.cuda.empty_cache()
    if qmm.device_status() != 0:
        raise RuntimeError("kernel reported a device-side error")
    out["how"] = ("CUDA-graph replay of >= 20 launches (one per weight copy, copies >= 4x L2), CUDA events "
                  "on the launching stream, median of 5 trials; us per launch")
    return out


def oracle_packed_layers():
    """Host copies of the six distinct layer matrices packed by the oracle's packer (the bytes
    qmm_pack writes, by the packers' byte-equality test), for the host-side baselines."""
    import numpy as np
    import oracle
    from bit_quantized_skinny_gb300 import inputs, workloads

    hosts = []
    for idx, (name, N, K) in enumerate(workloads.LAYER_SHAPES):
        buf = np.empty(N * (K // 256) * 144, dtype=np.uint8)
        rowbytes = (K // 256) * 144
        for row0, w in inputs.weight_chunks(N, K, inputs.seed_for(4, idx)):
            buf[row0 * rowbytes:(row0 + w.shape[0]) * rowbytes] = oracle.pack(w)
        hosts.append(buf)
    return hosts


def cpu_baseline(M: int, budget_s: float = 12.0):
    """The oracle as it stands, timed on the host cores over a bounded sample of the pass:
    evenly spaced rows of each of the six distinct matrices (packed by the oracle's packer), M
    activation rows, repeated until at least ~10 s of CPU work has run."""
    import numpy as np
    import oracle
    from bit_quantized_skinny_gb300 import inputs, workloads

    oracle.build()
    info = {"hosts": oracle_packed_layers()}
    cores = oracle.max_threads()
    shapes = workloads.LAYER_SHAPES
    xs = {K: inputs.activations_bf16_bits(M, K, 9) for K in {K for _, _, K in shapes}}
    # calibrate: time 2*cores rows of the down matrix
    t0 = time.perf_counter()
    N, K = shapes[5][1], shapes[5][2]
    oracle.matmul(info["hosts"][5], N, K, xs[K], rows=np.arange(2 * cores) % N)
    per_weight = (time.perf_counter() - t0) / (2 * cores * K)
    total_w = sum(N * K for _, N, K in shapes)
    frac = min(1.0, budget_s / (per_weight * total_w))
    done_bytes, t_total, sampled_rows, rounds = 0, 0.0, 0, 0
    while t_total < 0.8 * budget_s and rounds < 1000:
        for idx, (name, N, K) in enumerate(shapes):
            nrows = max(cores, int(N * frac))
            rows = np.linspace(0, N - 1, nrows).astype(np.int64)
            t0 = time.perf_counter()
            oracle.matmul(info["hosts"][idx], N, K, xs[K], rows=rows)
            t_total += time.perf_counter() - t0
            done_bytes += nrows * (K // 256) * 144
            sampled_rows += nrows
        rounds += 1
    # the same oracle on one thread, over a small sample of the down matrix (~2 s)
    N, K = shapes[5][1], shapes[5][2]
    n1 = max(1, int(2.0 / (per_weight * cores * K)))
    rows1 = np.linspace(0, N - 1, n1).astype(np.int64)
    t0 = time.perf_counter()
    oracle.matmul(info["hosts"][5], N, K, xs[K], rows=rows1, threads=1)
    t1 = time.perf_counter() - t0
    oracle.matmul(info["hosts"][5], N, K, xs[K], rows=rows1[:1], threads=cores)   # restores the thread count
    single = round(weight_gbps(n1 * (K // 256) * 144, t1 * 1e3), 4)
    return {"value": round(weight_gbps(done_bytes, t_total * 1e3), 4), "unit": UNIT, "cores": cores,
            "kind": "oracle", "single_thread_value": single,
            "sample": f"{rounds} round(s) over {sampled_rows // rounds} evenly spaced weight rows of the six "
                      f"distinct layer matrices ({done_bytes / 1e6:.1f} MB of packed weights in total, "
                      f"{frac * 100:.2f}% of one layer per round), M={M}, fp64, OpenMP over rows; {t_total:.1f} s; "
                      f"single_thread_value: {n1} rows of the down matrix on one thread, {t1:.1f} s"}


# ----------------------------------------------------------------------------- arms ------

def run_ours(args, rank: int, world: int, local_rank: int, dist_ok: bool):
    import numpy as np
    import torch
    from bit_quantized_skinny_gb300 import build_lib, qmm

    torch.cuda.set_device(local_rank)
    device = f"cuda:{local_rank}"
    if rank == 0:
        build_lib.build()
    sync = (lambda: torch.distributed.barrier()) if dist_ok else (lambda: None)
    sync()
    qmm.load()
    stream = torch.cuda.current_stream()
    M = args.M
    probes = peak_probes(device) if rank == 0 else None
    entries, info = layer_pass_setup(M, device)

    variant = qmm.select_variant_batched(entries, M)
    kernel = "q4k_tc_kernel" if variant == qmm.VARIANT_TC else "q4k_fma_kernel"
    # tensor cores: one activation-prep launch and one product launch per 160 matrices (their
    # tensor maps ride in the launch parameters); CUDA cores: one launch
    launches_per_step = (1 + -(-len(entries) // 160)) if variant == qmm.VARIANT_TC else 1
    step = lambda: qmm.run_batched(entries, M)
    step()
    torch.cuda.synchronize()
    if qmm.device_status() != 0:
        raise RuntimeError("kernel reported a device-side error")

    # five timed regions of exactly `steps` steps each; the step time is their median
    with ClockSampler(local_rank) as clocks:
        trials = time_trials(step, args.steps, args.warmup, stream, sync, trials=5)
    ms = statistics.median(trials)
    if qmm.device_status() != 0:
        raise RuntimeError("kernel reported a device-side error")
    wb = info["weight_bytes"]
    ms_max, wb_all = aggregate_ranks(ms, wb, dist_ok, device)
    per_gpu_gbps = GUARD.check(weight_gbps(wb, ms), "64-layer pass")
    value = weight_gbps(wb_all, ms_max)

    # ---- end to end through the C ABI with host buffers: H2D of X, the pass, D2H of Y
    pin_x = {K: x[0].cpu().pin_memory() for K, x in info["xs"].items()}
    pin_y = torch.empty(info["y_arena"].shape, dtype=torch.float32, pin_memory=True)
    h2d = sum(x.numel() * 2 for x in pin_x.values())
    d2h = pin_y.numel() * 4
    # The pass as calls of at most 160 products (the launches qmm_run_batched makes anyway); each
    # call's outputs (a contiguous range of the arena) go back to the host on a copy stream while
    # the next call computes.
    copy_stream = torch.cuda.Stream(device=device)
    parts = []
    for k0 in range(0, len(info["items"]), 160):
        its = info["items"][k0:k0 + 160]
        lo = sum(M * it[3] for it in info["items"][:k0])
        hi = lo + sum(M * it[3] for it in its)
        parts.append((qmm.make_entries(its), lo, hi))

    def e2e_step():
        for K, x in info["xs"].items():
            x[0].copy_(pin_x[K], non_blocking=True)
        for ents, lo, hi in parts:
            qmm.run_batched(ents, M)
            done = torch.cuda.Event()
            done.record(stream)
            copy_stream.wait_event(done)
            with torch.cuda.stream(copy_stream):
                pin_y[lo:hi].copy_(info["y_arena"][lo:hi], non_blocking=True)
        stream.wait_stream(copy_stream)   # the step ends when every output is on the host

    ms_e2e = statistics.median(time_trials(e2e_step, args.steps, args.warmup, stream, sync, trials=3))
    ms_e2e, _ = aggregate_ranks(ms_e2e, wb, dist_ok, device)
    GUARD.check(weight_gbps(wb, ms_e2e), "end-to-end pass")

    # ---- per-M sweep on the same pass (context for the switch point; same timing rules)
    per_m = {}
    if args.sweep and rank == 0:
        for m in args.sweep:
            ents_m, info_m = (entries, info) if m == M else layer_pass_setup(m, device)
            f = (lambda e=ents_m, mm=m: qmm.run_batched(e, mm))
            msm = statistics.median(time_trials(f, max(3, args.steps // 2), 3, stream, lambda: None, trials=3))
            g = GUARD.check(weight_gbps(info_m["weight_bytes"], msm), f"pass M={m}")
            per_m[str(m)] = {"gbps": round(g, 1), "ms_per_15.8GB_pass": round(ms_per_pass(g), 4),
                             "frac_of_measured_hbm": round(g / hbm_peak()[0], 4),
                             "frac_of_spec_8TBps": round(g / SPEC_HBM_GBS, 4),
                             "ms_per_row": round(msm / m, 4)}
            if m != M:
                del ents_m, info_m
                torch.cuda.empty_cache()

    peak, peak_kind = hbm_peak()
    achieved = info["algo_bytes"] / (ms * 1e-3) / 1e9
    algo_bytes = info["algo_bytes"]
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(M)
    # the other configurations, after the pass's buffers are released
    del entries, parts, pin_x, pin_y
    info_items = len(info["items"])
    info.clear()
    torch.cuda.empty_cache()
    configs = config_timings(device) if (rank == 0 and not args.no_configs) else None
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic: W ~ N(0, 0.02^2) packed to Q4K by qmm_pack, X ~ N(0,1) in bf16, seeded",
        "config": {
            "workload": "64-layer Q4K weight pass: per layer q 5120x5120, k 1024x5120, v 1024x5120, "
                        "o 5120x5120, gate_up 34816x5120, down 5120x17408 (384 matrices), "
                        f"M={M} bf16 rows, one qmm_run_batched call per pass",
            "M": M, "matrices": info_items, "weight_bytes_per_step": wb,
            "ms_per_15.8GB_pass": round(ms_per_pass(per_gpu_gbps), 4),
            "frac_of_spec_8TBps": round(per_gpu_gbps / SPEC_HBM_GBS, 4),
            "l2": "inputs larger than L2: 11.9 GB of weights per step vs 129 MB L2, no flush",
            "parallelism": f"{world} independent replica(s), one per GPU" if world > 1 else "1 GPU",
        },
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                     "traffic": recorded_traffic(kernel, "pass64", M),
                     "kernel": kernel,
                     "timed": "whole step on the launching stream (the product launches plus the "
                              "activation-prep launch, 0.15% of the step by ncu)" if variant == qmm.VARIANT_TC
                              else "whole step on the launching stream (one kernel)",
                     "algorithmic_bytes_per_step": algo_bytes,
                     "frac_of_read_probe": round(achieved / GUARD.read_gbps, 4) if GUARD.read_gbps else None,
                     "unit_of_measure": "one step = one qmm_run_batched call over the 384 matrices: one "
                                        "activation-prep launch and ceil(384/160) = 3 product launches; "
                                        "achieved and traffic are per step"},
        "e2e": {"value": round(weight_gbps(wb_all, ms_e2e), 2), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(ms_e2e, 5),
                "note": "qmm_run_batched with the step's X copied from pinned host memory and every "
                        "Y (one output arena) copied back to pinned host memory inside the timed "
                        "region, the pass as calls of at most 160 products whose outputs are copied "
                        "back on a second stream while the next call computes; the weights are "
                        "resident model parameters"},
        "gpu_launches": args.steps * launches_per_step,
        "timing": {"trials_ms_per_step": [round(t, 5) for t in trials], "statistic": "median of 5 timed regions "
                   "of exactly `steps` steps each (warm-up before the first)"},
        "peak_probes": probes,
        "configs": configs,
        "variant": qmm.VARIANT_NAMES.get(variant, str(variant)),
        "clocks": clocks.summary(),
        "per_M": per_m,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu
    if rank == 0:
        print(json.dumps(line), flush=True)


SINGLE_SHAPES = {"gate_up": (34816, 5120), "down": (5120, 17408), "q": (5120, 5120), "k": (1024, 5120),
                 "lm_head": (248320, 5120), "tiny": (256, 512)}


def run_profile_pass(args):
    """The small case that profiling captures: `--steps` steps of the pass over the first
    `--profile-pass` layers (one activation-prep launch and ceil(6 L / 160) product launches per
    step, all of them after `--warmup` warm-up steps), no timing.  Prints one JSON line."""
    import torch
    from bit_quantized_skinny_gb300 import build_lib, qmm

    build_lib.build()
    qmm.load()
    torch.cuda.set_device(0)
    layers = args.profile_pass
    entries, info = layer_pass_setup(args.M, "cuda", layers)
    for _ in range(args.warmup + args.steps):
        qmm.run_batched(entries, args.M)
    torch.cuda.synchronize()
    if qmm.device_status() != 0:
        raise RuntimeError("kernel reported a device-side error")
    print(json.dumps({"profile_pass": {"layers": layers, "matrices": len(entries), "M": args.M,
                                       "weight_bytes": info["weight_bytes"], "algorithmic_bytes": info["algo_bytes"],
                                       "steps": args.warmup + args.steps,
                                       "product_launches_per_step": -(-len(entries) // 160)}}), flush=True)


def run_single(args):
    """One product per launch, per shape x M x variant, weights cycled over copies totalling
    more than 4x L2 so every launch reads HBM.  Prints one JSON line."""
    import torch
    from bit_quantized_skinny_gb300 import build_lib, inputs, qmm, workloads

    build_lib.build()
    qmm.load()
    torch.cuda.set_device(0)
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    names = list(SINGLE_SHAPES)[:5] if args.single == "all" else [args.single]
    variants = {"fma": [qmm.VARIANT_FMA], "tc": [qmm.VARIANT_TC], "auto": [qmm.VARIANT_AUTO],
                "both": [qmm.VARIANT_FMA, qmm.VARIANT_TC]}[args.variant]
    stream = torch.cuda.current_stream()
    results = {}
    for name in names:
        N, K = SINGLE_SHAPES[name]
        Wd, _ = workloads.packed_weights(N, K, inputs.seed_for(3, list(SINGLE_SHAPES).index(name)), device="cuda")
        copies = max(1, -(-4 * l2 // Wd.numel()))
        ws = [Wd] + [Wd.clone() for _ in range(copies - 1)]
        res = {}
        for M in args.Ms:
            X, _ = workloads.activations(M, K, inputs.seed_for(3, 50 + M), device="cuda")
            Y = torch.empty((M, N), dtype=torch.float32, device="cuda")
            row = {"auto_picks": qmm.VARIANT_NAMES[qmm.select_variant(M, N, K)]}
            for v in variants:
                fn = lambda: [qmm.run(w, N, K, X, Y, M=M, variant=v) for w in ws]
                ms = time_steps(fn, max(2, args.steps // 5), 3, stream, lambda: None) / len(ws)
                row[qmm.VARIANT_NAMES.get(v, "auto")] = {"us": round(ms * 1e3, 2),
                                                         "gbps": round(weight_gbps(Wd.numel(), ms), 1)}
            res[str(M)] = row
            if qmm.device_status() != 0:
                raise RuntimeError("kernel reported a device-side error")
        results[name] = {"N": N, "K": K, "weight_bytes": Wd.numel(), "copies": copies, "per_M": res}
        del ws, Wd
        torch.cuda.empty_cache()
    print(json.dumps({"metric": "weight-read GB/s per single product (one launch each)", "unit": UNIT,
                      "l2": f"weights cycled over copies >= 4x L2 ({l2 >> 20} MB)", "shapes": results}), flush=True)


def run_ffn(args):
    """One feed-forward block per call (qmm_run_ffn: gate/up product, SiLU-gated bf16 step, down
    product) at the configurations' FFN shapes, weights cycled over copies totalling more than
    4x L2.  GB/s counts both matrices' packed weights.  Prints one JSON line."""
    import torch
    from bit_quantized_skinny_gb300 import build_lib, inputs, qmm, workloads

    build_lib.build()
    qmm.load()
    torch.cuda.set_device(0)
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    F, K = 17408, 5120
    Wgu, _ = workloads.packed_weights(2 * F, K, inputs.seed_for(2, 0), device="cuda")
    Wdn, _ = workloads.packed_weights(K, F, inputs.seed_for(2, 1), device="cuda")
    wbytes = Wgu.numel() + Wdn.numel()
    copies = max(1, -(-4 * l2 // wbytes))
    pairs = [(Wgu, Wdn)] + [(Wgu.clone(), Wdn.clone()) for _ in range(copies - 1)]
    stream = torch.cuda.current_stream()
    res = {}
    for M in args.Ms:
        X, _ = workloads.activations(M, K, inputs.seed_for(2, 50 + M), device="cuda")
        Y = torch.empty((M, K), dtype=torch.float32, device="cuda")
        ws = torch.empty(qmm.ffn_workspace_bytes(M, F), dtype=torch.uint8, device="cuda")
        fn = lambda: [qmm.run_ffn(g, d, F, K, X, Y, ws, M=M) for g, d in pairs]
        ms = time_steps(fn, max(2, args.steps // 5), 3, stream, lambda: None) / len(pairs)
        # the same calls captured once into a CUDA graph and replayed: no host work per block
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            fn()   # sizes the side stream's workspace before capture
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=side):
                fn()
        stream.wait_stream(side)
        ms_graph = time_steps(graph.replay, max(2, args.steps // 5), 3, stream, lambda: None) / len(pairs)
        # the fused block (gating in the gate/up epilogue; the weights read as row-interleaved:
        # the same bytes, so the same work)
        wsf = torch.empty(qmm.ffn_fused_workspace_bytes(M, F), dtype=torch.uint8, device="cuda")
        fnf = lambda: [qmm.run_ffn_fused(g, d, F, K, X, Y, wsf, M=M) for g, d in pairs]
        ms_f = time_steps(fnf, max(2, args.steps // 5), 3, stream, lambda: None) / len(pairs)
        with torch.cuda.stream(side):
            fnf()
            graph_f = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph_f, stream=side):
                fnf()
        stream.wait_stream(side)
        ms_fg = time_steps(graph_f.replay, max(2, args.steps // 5), 3, stream, lambda: None) / len(pairs)
        res[str(M)] = {"us": round(ms * 1e3, 2), "gbps": round(weight_gbps(wbytes, ms), 1),
                       "graph_us": round(ms_graph * 1e3, 2), "graph_gbps": round(weight_gbps(wbytes, ms_graph), 1),
                       "fused_us": round(ms_f * 1e3, 2), "fused_graph_us": round(ms_fg * 1e3, 2),
                       "fused_graph_gbps": round(weight_gbps(wbytes, ms_fg), 1),
                       "variants": [qmm.VARIANT_NAMES[qmm.select_variant(M, 2 * F, K)],
                                    qmm.VARIANT_NAMES[qmm.select_variant(M, K, F)]]}
        if qmm.device_status() != 0:
            raise RuntimeError("kernel reported a device-side error")
    print(json.dumps({"metric": "weight-read GB/s of one feed-forward block (gate/up -> SiLU gate -> down)",
                      "unit": UNIT, "F": F, "K": K, "weight_bytes": wbytes, "copies": copies,
                      "l2": f"weights cycled over copies >= 4x L2 ({l2 >> 20} MB)", "per_M": res}), flush=True)


def run_indexed(args):
    """The indexed-expert product (qmm_run_indexed) over 16 synthetic experts of 4096 x 5120
    (seeded, the same weight distribution as the other workloads), M rows spread over the experts
    round robin (M >= 16: every expert in use).  GB/s counts the packed weights of the experts in
    use (each read once per call); expert sets cycled over copies totalling more than 4x L2.
    Prints one JSON line."""
    import torch
    from bit_quantized_skinny_gb300 import build_lib, inputs, qmm, workloads

    build_lib.build()
    qmm.load()
    torch.cuda.set_device(0)
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    N, K, E = 4096, 5120, 16
    base, _ = workloads.packed_weights(N, K, inputs.seed_for(6, 0), device="cuda")
    experts = [base] + [base.clone() for _ in range(E - 1)]   # content does not change the timing
    ebytes = base.numel()
    copies = max(1, -(-4 * l2 // (ebytes * E)))
    sets = [experts] + [[w.clone() for w in experts] for _ in range(copies - 1)]
    stream = torch.cuda.current_stream()
    res = {}
    for M in args.Ms:
        ids = [i % E for i in range(M)]
        used = len(set(ids))
        X, _ = workloads.activations(M, K, inputs.seed_for(6, 50 + M), device="cuda")
        Y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        ws = torch.empty(qmm.indexed_workspace_bytes(M, N, K), dtype=torch.uint8, device="cuda")
        fn = lambda: [qmm.run_indexed(ex, N, K, ids, X, Y, ws) for ex in sets]
        ms = time_steps(fn, max(2, args.steps // 5), 3, stream, lambda: None) / len(sets)
        res[str(M)] = {"experts_used": used, "us": round(ms * 1e3, 2),
                       "gbps": round(weight_gbps(used * ebytes, ms), 1)}
        if qmm.device_status() != 0:
            raise RuntimeError("kernel reported a device-side error")
    print(json.dumps({"metric": "weight-read GB/s of the indexed-expert product (experts in use)", "unit": UNIT,
                      "experts": E, "N": N, "K": K, "expert_bytes": ebytes, "copies": copies,
                      "l2": f"expert sets cycled over copies >= 4x L2 ({l2 >> 20} MB)", "per_M": res}), flush=True)


def run_formats(args):
    """The other weight formats (Q5K, NVFP4 W4A16, INT4 with one scale per 128 columns) next
    to Q4K on the same tensor-core kernel: one product per launch, per format x shape x M,
    weights cycled over copies totalling more than 4x L2.  GB/s counts each format's packed
    bytes (its weight stream: what the launch must read).  Prints one JSON line."""
    import torch
    from bit_quantized_skinny_gb300 import build_lib, inputs, qmm, workloads

    build_lib.build()
    qmm.load()
    torch.cuda.set_device(0)
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    peak, _ = hbm_peak()
    names = ["gate_up", "down", "q", "lm_head"] if args.formats == "all" else args.formats.split(",")
    stream = torch.cuda.current_stream()
    results = {}
    fmts = qmm.FORMATS if not args.fmt else {k: qmm.FORMATS[k] for k in args.fmt.split(",")}
    for fname, fmt in fmts.items():
        per_shape = {}
        for name in names:
            N, K = SINGLE_SHAPES[name]
            Wd = workloads.packed_weights_fmt(fmt, N, K, inputs.seed_for(3, list(SINGLE_SHAPES).index(name)))
            copies = max(1, -(-4 * l2 // Wd.numel()))
            ws = [Wd] + [Wd.clone() for _ in range(copies - 1)]
            res = {}
            for M in args.Ms:
                X, _ = workloads.activations(M, K, inputs.seed_for(3, 50 + M), device="cuda")
                Y = torch.empty((M, N), dtype=torch.float32, device="cuda")
                if fmt == qmm.FMT_Q4K:   # the same tensor-core kernel as the other formats
                    fn = lambda: [qmm.run(w, N, K, X, Y, M=M, variant=qmm.VARIANT_TC) for w in ws]
                else:
                    fn = lambda: [qmm.fmt_run(fmt, w, N, K, X, Y, M=M) for w in ws]
                ms = time_steps(fn, max(2, args.steps // 5), 3, stream, lambda: None) / len(ws)
                gbps = weight_gbps(Wd.numel(), ms)
                res[str(M)] = {"us": round(ms * 1e3, 2), "gbps": round(gbps, 1),
                               "frac_of_measured_hbm": round(gbps / peak, 3)}
                if qmm.device_status() != 0:
                    raise RuntimeError("kernel reported a device-side error")
            per_shape[name] = {"N": N, "K": K, "weight_bytes": Wd.numel(),
                               "bits_per_weight": round(8 * Wd.numel() / (N * K), 4), "per_M": res}
            del ws, Wd
            torch.cuda.empty_cache()
        results[fname] = per_shape
    print(json.dumps({"metric": "weight-read GB/s per single product, by weight format", "unit": UNIT,
                      "peak_gbps": peak, "l2": f"weights cycled over copies >= 4x L2 ({l2 >> 20} MB)",
                      "formats": results}), flush=True)


def run_pass_formats(args):
    """The 64-layer pass (384 matrices) with its weights in each format, and a mixed pass
    (Q6K for the v and down projections, Q4K for the others: the pattern of the pages' Q4_K_M
    files, which mix k-quant widths), each as one qmm_fmt_run_batched call (one launch group per
    format present).  GB/s counts the packed bytes the pass reads.  Prints one JSON line."""
    import torch
    from bit_quantized_skinny_gb300 import build_lib, inputs, qmm, workloads

    build_lib.build()
    qmm.load()
    torch.cuda.set_device(0)
    peak, _ = hbm_peak()
    stream = torch.cuda.current_stream()
    plans = {name: (lambda shape, f=fmt: f) for name, fmt in qmm.FORMATS.items()}
    plans["mix_q4k_q6k"] = lambda shape: qmm.FMT_Q6K if shape in ("v", "down") else qmm.FMT_Q4K
    names = list(plans) if args.pass_formats == "all" else args.pass_formats.split(",")
    res = {}
    for pname in names:
        plan = plans[pname]
        for M in args.Ms:
            xs = {K: workloads.activations(M, K, inputs.seed_for(4, 100 + K % 97), device="cuda")[0]
                  for K in sorted({K for _, _, K in workloads.LAYER_SHAPES})}
            bases = {name: workloads.packed_weights_fmt(plan(name), N, K, inputs.seed_for(4, i))
                     for i, (name, N, K) in enumerate(workloads.LAYER_SHAPES)}
            items, keep = [], []
            for layer in range(LAYERS):
                for name, N, K in workloads.LAYER_SHAPES:
                    w = bases[name] if layer == 0 else bases[name].clone()
                    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
                    keep += [w, y]
                    items.append((plan(name), w, xs[K], y, N, K))
            entries = qmm.make_fmt_entries(items)
            wbytes = sum(it[1].numel() for it in items)
            fn = lambda: qmm.fmt_run_batched(entries, M)
            ms = time_steps(fn, max(3, args.steps // 2), 3, stream, lambda: None)
            g = weight_gbps(wbytes, ms)
            res[f"{pname}/M{M}"] = {"ms": round(ms, 4), "weight_bytes": wbytes, "gbps": round(g, 1),
                                    "frac_of_measured_hbm": round(g / peak, 4)}
            if qmm.device_status() != 0:
                raise RuntimeError("kernel reported a device-side error")
            del items, keep, bases, entries
            torch.cuda.empty_cache()
    print(json.dumps({"metric": "weight-read GB/s of the 64-layer pass by weight format", "unit": UNIT,
                      "peak_gbps": peak, "l2": "inputs larger than L2: every pass reads its weights from HBM",
                      "passes": res}), flush=True)


def run_reference(args, rank: int):
    """The oracle (plain fp64 C, host cores) on a bounded sample of the same workload."""
    if rank != 0:
        return
    import numpy as np
    import oracle
    from bit_quantized_skinny_gb300 import inputs, workloads

    oracle.build()
    cores = oracle.max_threads()
    M = args.M
    shapes = workloads.LAYER_SHAPES
    hosts = oracle_packed_layers()   # the oracle's packer: this arm loads nothing of the library
    xs = {K: inputs.activations_bf16_bits(M, K, 9) for K in {K for _, _, K in shapes}}
    # one step: a fixed, evenly spaced sample of rows from each distinct matrix (~1.5 s of work)
    N5, K5 = shapes[5][1], shapes[5][2]
    t0 = time.perf_counter()
    oracle.matmul(hosts[5], N5, K5, xs[K5], rows=np.arange(16 * cores) % N5)
    per_weight = (time.perf_counter() - t0) / (16 * cores * K5)
    total_w = sum(N * K for _, N, K in shapes)
    frac = min(1.0, 1.5 / (per_weight * total_w))
    samples = [np.linspace(0, N - 1, max(cores, int(N * frac))).astype(np.int64) for _, N, _ in shapes]
    step_bytes = sum(len(r) * (K // 256) * 144 for r, (_, _, K) in zip(samples, shapes))

    def step():
        for idx, (name, N, K) in enumerate(shapes):
            oracle.matmul(hosts[idx], N, K, xs[K], rows=samples[idx])

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    value = weight_gbps(step_bytes, dt * 1e3)
    sample = (f"{sum(len(r) for r in samples)} evenly spaced weight rows of the six distinct layer "
              f"matrices per step ({step_bytes / 1e6:.1f} MB packed), M={M}, fp64, OpenMP over rows")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic: W ~ N(0, 0.02^2) packed to Q4K, X ~ N(0,1) in bf16, seeded",
        "config": {"workload": "64-layer Q4K weight pass (bounded row sample per step), "
                               f"M={M}, the oracle on the host cores", "M": M},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--M", type=int, default=8)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--sweep", type=lambda s: [int(v) for v in s.split(",") if v], default=[1, 2, 4, 8, 16, 32])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the other configurations' graph-replay timings")
    ap.add_argument("--single", choices=list(SINGLE_SHAPES) + ["all"], default=None)
    ap.add_argument("--Ms", type=lambda s: [int(v) for v in s.split(",") if v], default=[1, 2, 3, 4, 7, 8, 9, 12, 16])
    ap.add_argument("--variant", choices=["fma", "tc", "auto", "both"], default="both")
    ap.add_argument("--ffn", action="store_true", help="time one feed-forward block per call instead")
    ap.add_argument("--indexed", action="store_true", help="time the indexed-expert product instead")
    ap.add_argument("--fmt", default=None, help="with --formats: only these formats (comma list)")
    ap.add_argument("--pass-formats", default=None,
                    help="time the 64-layer pass in these weight formats instead (comma list, 'mix_q4k_q6k' or 'all')")
    ap.add_argument("--profile-pass", type=int, default=0,
                    help="run warmup + steps steps of the first L layers' pass, untimed (the small case for ncu)")
    ap.add_argument("--formats", default=None,
                    help="time the weight formats on these shapes instead (comma list of gate_up,down,q,k,lm_head or 'all')")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if args.profile_pass:
        if rank == 0:
            run_profile_pass(args)
        return
    if args.single:
        if rank == 0:
            run_single(args)
        return
    if args.ffn:
        if rank == 0:
            run_ffn(args)
        return
    if args.indexed:
        if rank == 0:
            run_indexed(args)
        return
    if args.formats:
        if rank == 0:
            run_formats(args)
        return
    if args.pass_formats:
        if rank == 0:
            run_pass_formats(args)
        return
    dist_ok = False
    if world > 1:
        import torch
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        dist_ok = True
    try:
        run_ours(args, rank, world, local_rank, dist_ok)
    finally:
        if dist_ok:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
