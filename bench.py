#!/usr/bin/env python3
"""Benchmark of the RidgeFill upper-layer KV fill on GB300 (librf.so, C ABI).

One step = one rf_fill_kv call over the 27B-shaped workload (d=5120, L=64, S=16,
N=32768, T=4096, 8 KV heads x 128, 5% of prefix rows exact in blocks of 16, all
layers full attention): row compaction, gather, the map GEMM for all 48 upper
layers, the row RMS scales and the K/V GEMM with norm scale, RoPE and cache scatter. The RMSNorm
gains are folded into the projections once, before the timed region
(RF_WEIGHTS_PREFOLDED), and that fold is reported on its own. Inputs are seeded
synthetic tensors resident in HBM, larger than L2 (3.9 GB of maps, weights and x_S
are read per step), so no L2 flush is needed. Timing uses CUDA events on the
launching stream, bracketed by a barrier and a device synchronize.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 (under torchrun): the fill is sharded by upper layer: rank r fills its own
contiguous block of the upper layers (their maps, projections and cache slice),
with no data-path collective, so together the ranks fill the whole workload once
per step. value = all ranks' row-layers / max rank time (the only collective
reduces the timing numbers).
--impl reference times the fp64 CPU oracle on the host cores over a bounded row
sample of the same workload, and prints the same metric.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "filled rows×layers/s and fill TFLOP/s vs GB300 bf16 dense peak (1 GPU)"
UNIT = "row-layers/s"
WORKLOAD = "dense27b"
KERNELS_PER_FILL = 5   # compaction, gather, map GEMM, row RMS, K/V GEMM


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-rows", type=int, default=512, help="oracle row sample for the CPU baseline (all cores)")
    ap.add_argument("--cpu-rows-1core", type=int, default=16, help="oracle row sample for the single-core rate")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip timing the calibration, solve and cross-model rows")
    ap.add_argument("--extra", choices=EXTRA_ROWS, default=None,
                    help="time one row of the extras alone and print it (for short captures)")
    ap.add_argument("--capture-size", action="store_true",
                    help="with --extra: run a5_calibration with 4 maps and a7_xmodel with 12 -> 4 layers "
                         "(same per-unit work, a few GB on the device, for a full ncu capture)")
    ap.add_argument("--selection-only", action="store_true",
                    help="time only the source-selection row (all-source calibration + greedy selection)")
    ap.add_argument("--select-targets", type=int, default=0,
                    help="target layers for --selection-only (0 = the workload's 64; fewer for a short capture)")
    ap.add_argument("--select-sources", type=int, default=0,
                    help="source layers for --selection-only (0 = the workload's 40; fewer for a small capture)")
    ap.add_argument("--gemm", choices=["default", "single", "pair"], default="default",
                    help="tensor-core GEMM kernel: one CTA per 128x256 tile, or a CTA pair per 256x256 tile")
    ap.add_argument("--workload", choices=sorted(workloads()), default=WORKLOAD,
                    help="dense27b (default: the largest single-GPU workload); others for profiling runs")
    return ap.parse_args(argv)


def workloads():
    import dataclasses
    import synth
    w = dict(synth.FILL_CONFIGS)
    # ncu-sized case: 8B shapes, 8 upper layers, 4096 prefix rows (maps 268 MB > L2, ~1.5 GB on device)
    w["small"] = dataclasses.replace(synth.LLAMA8B, name="llama3.1-8b-shaped d4096 L20 S12 N4608 T512",
                                     L=20, S=12, N=4608, T=512)
    return w


# --------------------------------------------------------------------------- #
# Distributed plumbing (one process per GPU; timing reduction only)
# --------------------------------------------------------------------------- #
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return ws, rank, local


def dist_init(backend: str):
    import torch.distributed as dist
    ws, rank, _ = dist_env()
    if ws > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        os.environ.setdefault("MASTER_PORT", "29511")
        dist.init_process_group(backend=backend, rank=rank, world_size=ws)
    return ws, rank


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def reduce_max(x: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(x: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def aggregate_timing(units_per_step: float, steps: int, elapsed_ms: float, device=None):
    """Whole-job throughput: every rank's units over the slowest rank's time.
    Returns (value per second, ms per step, max elapsed ms)."""
    t_max = reduce_max(elapsed_ms, device)
    total = reduce_sum(float(units_per_step) * steps, device)
    return total / (t_max / 1e3), t_max / steps, t_max


# --------------------------------------------------------------------------- #
# Clock sampling during the timed region
# --------------------------------------------------------------------------- #
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="rf_clocks_", suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) >= 10:
                    rows.append(p)
        os.unlink(self.path)
        if not rows:
            return None

        def num(s):
            try:
                return float(s)
            except ValueError:
                return None
        load = [r for r in rows if (num(r[4]) or 0) >= 50] or rows
        sm = [num(r[1]) for r in load if num(r[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in load for i in range(4) if r[6 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": num(load[0][2]), "reasons": reasons, "samples": len(load),
                "power_w_max": max((num(r[3]) or 0) for r in load)}


# --------------------------------------------------------------------------- #
# Helpers
# --------------------------------------------------------------------------- #
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return {"hbm_gbs": j.get("hbm_gbs"), "bf16_tflops": j.get("bf16_tflops"),
                "bf16_tflops_sustained": j.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# The sources the fill GEMMs are compiled from (their kernels are instantiated in
# fill.cu only); a committed DRAM-traffic figure is valid while these hash the same.
FILL_GEMM_SOURCES = ("api.cu", "epilogue.cuh", "fill.cu", "fill_gemm.cuh", "rf_device.cuh", "rf_host.h",
                     "tc_gemm.cuh")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.json")


def kernel_source_sha() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "ridge_map_kv_gb300", "csrc")
    for f in FILL_GEMM_SOURCES:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + b"\0" + fh.read())
    h.update(b"rf.h\0" + open(os.path.join(ROOT, "include", "rf.h"), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of ``kernel`` on ``workload`` from the machine-readable
    record written with the ncu capture (profiles/dram_traffic.json), if it was taken
    on the current kernel sources; else None."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        rec = json.load(f).get(f"{kernel}/{workload}")
    if not rec or rec.get("source_sha") != kernel_source_sha():
        return None
    return float(rec["bytes_per_launch"])


def fill_units(cfg, mask):
    n_prefix = cfg.N - cfg.T
    n_fill = n_prefix - (int(mask.sum().item()) if mask is not None else 0)
    return n_fill, n_fill * cfg.P


class OracleInputs:
    """The workload's tensors decoded once to float64 (bf16 decoding is exact and
    is input marshalling, not the oracle's arithmetic)."""

    def __init__(self, cfg, inp):
        import numpy as np
        import oracle as O
        import synth
        f64 = O.bf16_bits_to_f64
        self.cfg = cfg
        mask = None if inp["mask"] is None else inp["mask"].cpu().numpy()
        self.idx = O.prefix_partition(cfg.N, cfg.T, mask)
        self.x = f64(synth.bits(inp["x_S"]))
        self.A = [f64(synth.bits(inp["A"][p:p + 1])) for p in range(cfg.P)]
        self.b = [synth.f32(inp["b"][p:p + 1]).astype(np.float64) for p in range(cfg.P)]
        self.g = [f64(synth.bits(inp["gain"][p:p + 1])) for p in range(cfg.P)]
        self.Wk = [f64(synth.bits(inp["Wk"][p:p + 1])) for p in range(cfg.P)]
        self.Wv = [f64(synth.bits(inp["Wv"][p:p + 1])) for p in range(cfg.P)]


def cpu_oracle_rate(oi: "OracleInputs", n_rows: int, seed: int = 7):
    """Times the fp64 oracle (fill_rows, all upper layers) on ``n_rows`` filled rows."""
    import numpy as np
    import oracle as O
    cfg = oi.cfg
    rows = np.sort(np.random.default_rng(seed).choice(oi.idx, size=min(n_rows, len(oi.idx)), replace=False))
    t0 = time.perf_counter()
    x = oi.x[rows]
    for p in range(cfg.P):
        O.fill_rows(x, rows + cfg.pos_offset, oi.A[p], oi.b[p], oi.g[p], oi.Wk[p], oi.Wv[p],
                    cfg.H, cfg.hd, cfg.rope_theta, cfg.rms_eps)
    dt = time.perf_counter() - t0
    return len(rows) * cfg.P / dt, dt, len(rows), host_cores()


def host_cores() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()


class BlasThreads:
    """Thread count of the BLAS library numpy loaded (OpenBLAS builds export a
    set/get pair), so the oracle can be timed on one core. ``available`` is False
    when no such library is found; nothing is changed then."""
    PAIRS = (("scipy_openblas_get_num_threads64_", "scipy_openblas_set_num_threads64_"),
             ("openblas_get_num_threads64_", "openblas_set_num_threads64_"),
             ("openblas_get_num_threads", "openblas_set_num_threads"))

    def __init__(self):
        import ctypes

        import numpy as np
        np.ones((2, 2)) @ np.ones((2, 2))          # make sure the BLAS library is loaded
        self.get = self.set = None
        paths = []
        with open("/proc/self/maps") as f:
            for line in f:
                if "blas" in line.lower() and line.split()[-1] not in paths:
                    paths.append(line.split()[-1])
        for path in paths:
            try:
                lib = ctypes.CDLL(path)
            except OSError:
                continue
            for g, s_ in self.PAIRS:
                if hasattr(lib, g) and hasattr(lib, s_):
                    self.get, self.set = getattr(lib, g), getattr(lib, s_)
                    self.get.restype = ctypes.c_int
                    self.set.argtypes = [ctypes.c_int]
                    return

    @property
    def available(self) -> bool:
        return self.set is not None


def cpu_baseline(cfg, inp, n_rows: int, n_rows_1core: int) -> dict:
    """The fp64 oracle as it stands, on this host: all cores on ``n_rows`` sampled
    filled rows x every upper layer, one core on ``n_rows_1core`` rows, and the
    whole toy workload (every filled row and layer of the 8-layer toy) once."""
    import numpy as np

    import oracle as O
    import synth
    oi = OracleInputs(cfg, inp)
    rate, dt, nrows, cores = cpu_oracle_rate(oi, n_rows)
    out = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
           "sample": f"{nrows} filled rows x {cfg.P} upper layers of the same workload, fp64 numpy, {dt:.1f} s"}
    bt = BlasThreads()
    if bt.available:
        before = bt.get()
        bt.set(1)
        try:
            r1, dt1, n1, _ = cpu_oracle_rate(oi, n_rows_1core, seed=8)
        finally:
            bt.set(before)
        out["single_core"] = {"value": r1, "unit": UNIT, "cores": 1,
                              "sample": f"{n1} filled rows x {cfg.P} upper layers, BLAS on one thread, {dt1:.1f} s"}
    else:
        out["single_core"] = {"value": None, "why": "no OpenBLAS thread control found in this numpy"}
    toy = synth.TOY
    ti = synth.fill_inputs(toy)
    f64 = O.bf16_bits_to_f64
    zeros = np.zeros((toy.L, toy.N, toy.H, toy.hd))
    t0 = time.perf_counter()
    O.fill_kv(zeros, zeros, f64(synth.bits(ti["x_S"])), synth.f32(ti["mask"]), f64(synth.bits(ti["A"])),
              synth.f32(ti["b"]).astype(np.float64), f64(synth.bits(ti["gain"])), f64(synth.bits(ti["Wk"])),
              f64(synth.bits(ti["Wv"])), L=toy.L, S=toy.S, N=toy.N, T=toy.T, n_kv_heads=toy.H, head_dim=toy.hd,
              rope_theta=toy.rope_theta, rms_eps=toy.rms_eps)
    out["toy_full_s"] = time.perf_counter() - t0
    out["toy_workload"] = f"{toy.name}: the whole fill (every filled row and upper layer, bookkeeping included)"
    del oi
    return out


def gemm_flags(name):
    """RF_FLAG_* bits for the --gemm choice (0 = the library's default kernel)."""
    return {"default": 0, "single": 1, "pair": 2}[name]


# --------------------------------------------------------------------------- #
# Our arm
# --------------------------------------------------------------------------- #
def run_extra_only(args):
    import json

    import torch
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peaks = measured_peaks()
    print(json.dumps(run_extras(dev, peaks["bf16_tflops"], gemm_flags(args.gemm), only=args.extra,
                                capture=args.capture_size)))


def run_selection_only(args):
    import json

    import torch
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peaks = measured_peaks()
    row = run_selection(dev, peaks["bf16_tflops"], gemm_flags(args.gemm), args.select_targets, args.select_sources)
    print(json.dumps({"selection": row}))


def fill_plan(cfg, world: int, rank: int, flags: int):
    """The rank's share of the fill: its layer block and the rf_fill_desc fields of
    that block (see ridge_map_kv_gb300.shard). One rank covers the whole fill."""
    from ridge_map_kv_gb300 import shard as sh
    block = sh.layer_shard(cfg.P, cfg.S, world, rank)
    fields = dict(d=cfg.d, d_in=cfg.d_in, L=cfg.L, S=cfg.S, N=cfg.N, T=cfg.T, n_kv_heads=cfg.H, head_dim=cfg.hd,
                  rope_theta=cfg.rope_theta, rms_eps=cfg.rms_eps, pos_offset=cfg.pos_offset, flags=flags)
    return block, sh.shard_desc_fields(fields, block)


def run_ours(args):
    import torch

    import ridge_map_kv_gb300 as rf
    import synth
    from ridge_map_kv_gb300 import shard as sh

    ws_n, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist_init("nccl")
    dev = torch.device("cuda", local)
    cfg = workloads()[args.workload]
    full = synth.fill_inputs(cfg, device=dev)
    n_fill, _ = fill_units(cfg, full["mask"])
    block, fields = fill_plan(cfg, ws_n, rank, gemm_flags(args.gemm) | rf.RF_WEIGHTS_PREFOLDED)
    inp = sh.shard_weights(full, block)
    P, d, KV, di = block.layers, cfg.d, cfg.KV, cfg.D_in
    units = n_fill * P
    desc = rf.rf_fill_desc(**fields)
    kc = torch.zeros((max(P, 1), cfg.N, cfg.H, cfg.hd), dtype=torch.bfloat16, device=dev)   # this rank's layers
    vc = torch.zeros_like(kc)
    ws_bytes = rf.rf_fill_workspace_bytes(desc)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    nfill = torch.zeros(1, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    # one-time weight preparation (reported separately, outside the step)
    Wk = torch.empty_like(inp["Wk"])
    Wv = torch.empty_like(inp["Wv"])
    rf.rf_profile_start(8)
    rf.rf_fold_kv_weights(desc, inp["gain"], inp["Wk"], inp["Wv"], Wk, Wv)
    fold_ms = sum(ms for _, ms in rf.rf_profile_stop())

    def step():
        rf.rf_fill_kv(desc, inp["x_S"], di, inp["mask"], inp["A"], inp["b"], None, Wk, Wv, kc, vc, cfg.N * KV, KV,
                      nfill, status, ws, ws_bytes)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    assert int(nfill.item()) == n_fill

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.4)                      # let the sampler start before the timed region
    cap = args.steps * KERNELS_PER_FILL + 64
    rf.rf_profile_start(cap)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    prof = rf.rf_profile_stop(cap)
    elapsed_ms = e0.elapsed_time(e1)
    assert int(status.item()) == 0
    assert len(prof) < cap, "profiler capacity reached: launch count would be cut short"
    value, ms_per_step, t_max = aggregate_timing(units, args.steps, elapsed_ms, dev)

    stage_ms = {}
    for name, ms in prof:
        stage_ms.setdefault(name, []).append(ms)
    stage_avg = {k: sum(v) / len(v) for k, v in stage_ms.items()}
    launches = len(prof)

    map_flops = 2.0 * n_fill * P * d * di
    kv_flops = 2.0 * n_fill * P * d * 2 * KV
    fill_flops_rank = map_flops + kv_flops
    fill_flops_all = reduce_sum(fill_flops_rank, dev)
    peaks = measured_peaks()
    # The GEMMs are timed inside the whole run of K steps: a run of 0.2 s or more is
    # a sustained load (the 1.4 kW power cap engages within it), so the denominator
    # is the sustained bf16 figure; a shorter run takes the burst one. Both fractions
    # are in the line.
    sustained = t_max >= 200.0 and peaks.get("bf16_tflops_sustained")
    peak = peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"]
    m_pad = -(-n_fill // 256) * 256

    def roofline_of(stage, kernel, flops, nbytes, traffic_key):
        ms_k = stage_avg.get(stage)
        achieved = flops / (ms_k / 1e3) / 1e12 if ms_k else None
        return {"kernel": kernel, "bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": (achieved / peak) if achieved else None,
                "frac_of_burst": (achieved / peaks["bf16_tflops"]) if achieved else None,
                "traffic": profiled_traffic(traffic_key, args.workload) if ws_n == 1 else None,
                "peak_source": f"{peaks['source']} {'sustained' if sustained else 'burst'} bf16 (MEASURED_PEAKS.json)"
                               f"; timed region {t_max:.0f} ms",
                "peak_burst": peaks["bf16_tflops"], "peak_sustained": peaks.get("bf16_tflops_sustained"),
                "ms_per_launch": ms_k, "algorithmic_flops_per_launch": flops, "algorithmic_bytes_per_launch": nbytes}

    # algorithmic bytes: map GEMM = Xf + maps + x̂ + Σx̂² partials + b; K/V GEMM = x̂ + Wk/Wv + the cache rows
    map_bytes = n_fill * di * 2 + P * d * di * 2 + n_fill * P * d * 2 + n_fill * P * (d // 256) * 4 + P * d * 4
    kv_bytes = n_fill * P * d * 2 + P * 2 * KV * d * 2 + n_fill * P * 2 * KV * 2
    roofline = roofline_of("map_gemm", "map_gemm (tc_gemm_pair_kernel<MapProb>)", map_flops, map_bytes, "map_gemm")
    roofline_kv = roofline_of("kv_gemm", "kv_gemm (tc_gemm_pair_kernel<KVProb>)", kv_flops, kv_bytes, "kv_gemm")

    # HBM-bound kernels of the step against the measured copy bandwidth:
    # gather = read n_fill rows of x_S + write Xf (n_fill rows, zero pad to the
    # 256-row unit); compaction = read the mask + write fill_idx; row_rms = read
    # the map GEMM's d/256 partial sums per row and layer + write the row scale.
    n_prefix = cfg.N - cfg.T
    hbm_bytes = {"gather": n_fill * di * 2 + m_pad * di * 2,
                 "compact": n_prefix + n_fill * 4,
                 "row_rms": P * (d // 256) * n_fill * 4 + P * n_fill * 4}
    hbm_kernels = {}
    for k, nbytes in hbm_bytes.items():
        ms_k = stage_avg.get(k)
        if ms_k:
            gbs = nbytes / (ms_k / 1e3) / 1e9
            hbm_kernels[k] = {"bytes": nbytes, "ms": ms_k, "GB/s": gbs, "frac": gbs / peaks["hbm_gbs"],
                              "peak": peaks["hbm_gbs"], "peak_source": f"{peaks['source']} copy (MEASURED_PEAKS.json)"}

    # End to end through the C ABI from pinned host buffers: every step copies
    # x_S and the mask host->device and reads n_fill and the status word back.
    # The copies run on a second stream into two device buffers, so step i+1's
    # inputs travel while step i computes (events order each buffer's reuse);
    # the first copy starts after the opening event and the last read-back ends
    # before the closing one, so all of it is inside the timed region.
    e2e = None
    if not args.no_e2e:
        xh = inp["x_S"].cpu().pin_memory()
        has_mask = inp["mask"] is not None
        mh = inp["mask"].cpu().pin_memory() if has_mask else torch.zeros(0, dtype=torch.uint8)
        xd = [torch.empty_like(inp["x_S"]) for _ in range(2)]
        md = [torch.empty_like(inp["mask"]) if has_mask else None for _ in range(2)]
        outh = torch.zeros(2, dtype=torch.int32).pin_memory()
        outd = torch.zeros(2, dtype=torch.int32, device=dev)
        copy_stream = torch.cuda.Stream(device=dev)
        ready = [torch.cuda.Event() for _ in range(2)]
        freed = [torch.cuda.Event() for _ in range(2)]

        def run_e2e(n_steps, start_event=None):
            if start_event is not None:
                copy_stream.wait_event(start_event)
            for i in range(n_steps):
                r = i & 1
                with torch.cuda.stream(copy_stream):
                    if i >= 2:
                        copy_stream.wait_event(freed[r])
                    xd[r].copy_(xh, non_blocking=True)
                    if has_mask:
                        md[r].copy_(mh, non_blocking=True)
                    ready[r].record(copy_stream)
                stream.wait_event(ready[r])
                rf.rf_fill_kv(desc, xd[r], di, md[r], inp["A"], inp["b"], None, Wk, Wv, kc, vc, cfg.N * KV, KV,
                              outd[0:1], outd[1:2], ws, ws_bytes, stream=stream.cuda_stream)
                freed[r].record(stream)
                outh.copy_(outd, non_blocking=True)
        run_e2e(3)
        torch.cuda.synchronize()
        barrier()
        e0.record(stream)
        run_e2e(args.steps, start_event=e0)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        assert int(outh[0]) == n_fill and int(outh[1]) == 0
        e2e_value, e2e_ms, _ = aggregate_timing(units, args.steps, e0.elapsed_time(e1), dev)
        e2e = {"value": e2e_value, "unit": UNIT,
               "h2d_bytes_per_step": xh.numel() * 2 + mh.numel(), "d2h_bytes_per_step": 8,
               "ms_per_step": e2e_ms, "copies": "pinned host -> device on a second stream, double-buffered"}

    cpu = None
    if rank == 0 and ws_n == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(cfg, full, args.cpu_rows, args.cpu_rows_1core)

    extras = None
    if rank == 0 and ws_n == 1 and not args.no_extras:
        del ws, kc, vc, inp, full, Wk, Wv
        torch.cuda.empty_cache()
        extras = run_extras(dev, peaks["bf16_tflops"], gemm_flags(args.gemm))

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws_n, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "strong" if ws_n > 1 else "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": workload_label(cfg), "n_fill": n_fill,
                       "upper_layers": cfg.P, "row_layers_per_step": n_fill * cfg.P,
                       "parallelism": f"upper layers sharded over {ws_n} GPU(s), {block.layers} layers on rank 0"
                                      if ws_n > 1 else "1 GPU, whole fill",
                       "gemm": args.gemm, "weights": "RMSNorm gain folded into W_k/W_v once, before the timed "
                                                     "region (RF_WEIGHTS_PREFOLDED); fold_once_ms",
                       "l2": "no flush: inputs larger than L2 (maps, projections and x_S read per step)"},
            "tflops": fill_flops_all * args.steps / (t_max / 1e3) / 1e12,
            "frac_of_bf16_peak": fill_flops_all * args.steps / (t_max / 1e3) / 1e12 / peak,
            "roofline": roofline, "roofline_kv_gemm": roofline_kv, "hbm_kernels": hbm_kernels,
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches, "clocks": clk,
            "stages_ms": stage_avg, "fold_once_ms": fold_ms, "extras": extras,
        }
        print(json.dumps(line))


def workload_label(cfg) -> str:
    exact = {None: "no exact prefix rows", "uniform10": "10% exact prefix rows (uniform)",
             "blocks16_5": "5% exact prefix rows in blocks of 16"}.get(cfg.exact, f"exact rows {cfg.exact}")
    return f"{cfg.name}, {cfg.H}x{cfg.hd} KV heads, {exact}"


# --------------------------------------------------------------------------- #
# The other rows of the path, timed once each at their workloads' sizes
# --------------------------------------------------------------------------- #
def _timed(fn, reps, stream):
    import torch
    import ridge_map_kv_gb300 as rf
    fn()
    torch.cuda.synchronize()
    rf.rf_profile_start(4096)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    stages = {}
    for name, ms in rf.rf_profile_stop():
        stages[name] = stages.get(name, 0.0) + ms / reps
    return e0.elapsed_time(e1) / reps, stages


def _prefolded(c, inp, flags):
    """rf_fill_desc of workload ``c`` with RF_WEIGHTS_PREFOLDED, and its folded K/V
    projections (the unfolded ones are dropped from ``inp``)."""
    import torch

    import ridge_map_kv_gb300 as rf
    fd = rf.rf_fill_desc(d=c.d, d_in=c.d_in, L=c.L, S=c.S, N=c.N, T=c.T, n_kv_heads=c.H, head_dim=c.hd,
                         rope_theta=c.rope_theta, rms_eps=c.rms_eps, pos_offset=0, flags=flags | rf.RF_WEIGHTS_PREFOLDED)
    Wk, Wv = torch.empty_like(inp["Wk"]), torch.empty_like(inp["Wv"])
    rf.rf_fold_kv_weights(fd, inp["gain"], inp["Wk"], inp["Wv"], Wk, Wv)
    del inp["Wk"], inp["Wv"]
    return fd, Wk, Wv


def _zero_stats(d_in, d_out, P, dev):
    import torch
    return {"G": torch.zeros((d_in, d_in), dtype=torch.float64, device=dev),
            "C": torch.zeros((P, d_in, d_out), dtype=torch.float64, device=dev),
            "sx": torch.zeros(d_in, dtype=torch.float64, device=dev),
            "sy": torch.zeros((P, d_out), dtype=torch.float64, device=dev),
            "n": torch.zeros(1, dtype=torch.int64, device=dev)}


EXTRA_ROWS = ("fill_llama8b", "a5_calibration", "a5_calibration_xmodel", "a6_solve", "a6_solve_27b",
              "a6_solve_xmodel", "a7_xmodel", "next3_map_storage_8b", "next3_map_storage_27b",
              "next2_key_norm_qwen3", "next4_nonsquare_flash_next", "next1_value_rescale_27b",
              "next4a_source_selection_xmodel")


def run_extras(dev, peak_tflops, flags=0, only=None, capture=False):
    """The other rows of the path, each timed with CUDA events at its workload's
    size: calibration (27B shape, and the cross-model Gram), the ridge solve (8B
    shape, 20 maps), the cross-model mapper (40 -> 64 layers, N = 32768), the NEXT
    rows and the source selection. `only` names one row (EXTRA_ROWS) to run alone.
    `capture` shrinks the 27B calibration to 4 maps and the mapper to 12 -> 4
    layers: the same units at a size a full ncu capture can save and restore."""
    import torch

    import ridge_map_kv_gb300 as rf
    import synth
    stream = torch.cuda.current_stream(dev)
    out = {}

    if only in (None, "fill_llama8b"):
        # the Llama-3.1-8B-shaped fill (20 upper layers, n_fill = 11,059), weights prefolded
        c = synth.LLAMA8B
        inp = synth.fill_inputs(c, device=dev)
        fd, Wk, Wv = _prefolded(c, inp, flags)
        kc = torch.zeros((c.L, c.N, c.KV), dtype=torch.bfloat16, device=dev)
        vc = torch.zeros_like(kc)
        wsb = rf.rf_fill_workspace_bytes(fd)
        ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
        nf = torch.zeros(1, dtype=torch.int32, device=dev)
        ms, st = _timed(lambda: rf.rf_fill_kv(fd, inp["x_S"], c.d, inp["mask"], inp["A"], inp["b"], None, Wk, Wv, kc,
                                              vc, c.N * c.KV, c.KV, nf, None, ws, wsb), 20, stream)
        n_fill = int(nf.item())
        f_flops = 2.0 * n_fill * c.P * (c.d * c.d + c.d * 2 * c.KV)
        mg, kg = st.get("map_gemm"), st.get("kv_gemm")
        out["fill_llama8b"] = {
            "workload": workload_label(c) + f", n_fill={n_fill}", "fill_ms": ms,
            "fill_row_layers_per_s": n_fill * c.P / (ms / 1e3), "fill_tflops": f_flops / (ms / 1e3) / 1e12,
            "fill_frac_of_bf16_peak": f_flops / (ms / 1e3) / 1e12 / peak_tflops,
            "map_gemm_frac_of_bf16_peak": 2.0 * n_fill * c.P * c.d * c.d / (mg / 1e3) / 1e12 / peak_tflops if mg else None,
            "kv_gemm_frac_of_bf16_peak": 2.0 * n_fill * c.P * c.d * 2 * c.KV / (kg / 1e3) / 1e12 / peak_tflops
            if kg else None, "stages_ms": st}
        del inp, kc, vc, ws, Wk, Wv
        torch.cuda.empty_cache()

    if only in (None, "a5_calibration"):
        # a5: calibration statistics, 27B-shaped: XᵀX and XᵀY_l for 48 maps over 16,384 rows
        c = synth.DENSE27B
        d, P, n = c.d, (4 if capture else c.P), c.calib_n
        cal = synth.calib_inputs(d, d, P, n, index=c.index, device=dev)
        st = _zero_stats(d, d, P, dev)
        cs = rf.calib_stats_struct(st["G"], st["C"], st["sx"], st["sy"], st["n"])
        cd = rf.rf_calib_desc(d_in=d, d_out=d, n_maps=P, flags=flags)
        cw = torch.empty(rf.rf_calib_workspace_bytes(cd, n), dtype=torch.uint8, device=dev)
        ms, stages = _timed(lambda: rf.rf_calib_accumulate(cd, cal["X"], d, cal["Y"], d, n * d, n, cs, None, cw,
                                                           cw.numel()), 3, stream)
        ms_fixed, st_fixed = _timed(lambda: rf.rf_calib_accumulate(cd, cal["X"], d, cal["Y"], d, n * d, n, cs), 3, stream)
        # algorithmic flops: XᵀX is symmetric, so its upper triangle (with the diagonal), plus every XᵀY_l
        flops = 1.0 * n * d * (d + 1) + 2.0 * n * d * d * P
        gm = stages.get("calib_gemm", ms)
        out["a5_calibration"] = {
            "workload": f"27b-shaped XᵀX + XᵀY, d={d}, {P} maps, {n} rows per call",
            "ms_per_call": ms, "tflops": flops / (ms / 1e3) / 1e12, "gemm_ms": gm,
            "gemm_frac_of_bf16_peak": flops / (gm / 1e3) / 1e12 / peak_tflops, "stages_ms": stages,
            "gemm_ms_round_robin_order": st_fixed.get("calib_gemm", ms_fixed)}
        del cal, st, cs
        torch.cuda.empty_cache()

    if only in (None, "a5_calibration_xmodel"):
        # a5, cross-model: the 8192-feature Gram over 131,072 rows and XᵀY for one target layer (1024 columns)
        x = synth.XMODEL
        d_in, d_out, n = x.d_in, x.KV, x.calib_n
        cal = synth.calib_inputs(d_in, d_out, 1, n, index=x.index, device=dev)
        st = _zero_stats(d_in, d_out, 1, dev)
        cs = rf.calib_stats_struct(st["G"], st["C"], st["sx"], st["sy"], st["n"])
        cd = rf.rf_calib_desc(d_in=d_in, d_out=d_out, n_maps=1, flags=flags)
        cw = torch.empty(rf.rf_calib_workspace_bytes(cd, n), dtype=torch.uint8, device=dev)
        ms, stages = _timed(lambda: rf.rf_calib_accumulate(cd, cal["X"], d_in, cal["Y"], d_out, n * d_out, n, cs,
                                                           None, cw, cw.numel()), 3, stream)
        ms_fixed, st_fixed = _timed(lambda: rf.rf_calib_accumulate(cd, cal["X"], d_in, cal["Y"], d_out, n * d_out, n,
                                                                   cs), 3, stream)
        flops = 1.0 * n * d_in * (d_in + 1) + 2.0 * n * d_in * d_out
        gm = stages.get("calib_gemm", ms)
        out["a5_calibration_xmodel"] = {
            "workload": f"cross-model calibration: XᵀX over d_in={d_in} features and XᵀY for {d_out} target columns, "
                        f"{n} rows per call",
            "ms_per_call": ms, "tflops": flops / (ms / 1e3) / 1e12, "gemm_ms": gm,
            "gemm_frac_of_bf16_peak": flops / (gm / 1e3) / 1e12 / peak_tflops, "stages_ms": stages,
            "gemm_ms_round_robin_order": st_fixed.get("calib_gemm", ms_fixed)}
        del cal, st, cs
        torch.cuda.empty_cache()

    if only in (None, "a6_solve"):
        # a6: ridge solve, 8B-shaped (d = 4096, 20 maps) from 8192 calibration rows
        c = synth.LLAMA8B
        d, P, n = c.d, c.P, c.calib_n
        cal = synth.calib_inputs(d, d, P, n, index=c.index, device=dev)
        st = _zero_stats(d, d, P, dev)
        cs = rf.calib_stats_struct(st["G"], st["C"], st["sx"], st["sy"], st["n"])
        cd = rf.rf_calib_desc(d_in=d, d_out=d, n_maps=P, flags=flags)
        rf.rf_calib_accumulate(cd, cal["X"], d, cal["Y"], d, n * d, n, cs)
        del cal
        A = torch.empty((P, d, d), dtype=torch.float32, device=dev)
        b = torch.empty((P, d), dtype=torch.float32, device=dev)
        Ab = torch.empty((P, d, d), dtype=torch.bfloat16, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        wsb = rf.rf_solve_workspace_bytes(cd)
        ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
        sol = {}
        for refine in (0, 1):
            ms, stages = _timed(lambda: rf.rf_solve(cd, cs, c.lam, rf.RF_ALPHA_TRACE, refine, A, b, Ab, None, status,
                                                   ws, wsb), 1, stream)
            sol[f"refine_{refine}_ms"] = ms
            sol[f"refine_{refine}_stages_ms"] = stages
        assert int(status.item()) == 0
        # A_p = Cc_pᵀ H^-1: 2 P d³ fp32-accurate flops, as six bf16 plane products each
        prod = 2.0 * P * d ** 3
        pm = sol["refine_0_stages_ms"].get("solve_product")
        if pm:
            sol["product_bf16_plane_tflops"] = 6.0 * prod / (pm / 1e3) / 1e12
            sol["product_frac_of_bf16_peak"] = sol["product_bf16_plane_tflops"] / peak_tflops
        # one refinement sweep: the residual A_p H as 21 digit-pair products (6 digits a side,
        # weights s + t <= 7) plus the correction R_p H^-1 (six plane products)
        rm = sol["refine_1_stages_ms"].get("solve_refine")
        if rm:
            # one sweep = the residual A_p H plus the correction R_p H^-1: 2 products of the
            # solve's size, fp64-accurate and fp32-accurate (how many bf16 digit and plane
            # products that takes depends on the conditioning the library estimates)
            sol["refine_sweep_ms"] = rm
            sol["refine_product_equiv_tflops"] = 2.0 * prod / (rm / 1e3) / 1e12
        out["a6_solve"] = {"workload": f"8b-shaped ridge solve, d={d}, {P} maps, lambda={c.lam}", **sol}
        del st, cs, A, b, Ab, ws
        torch.cuda.empty_cache()

    if only in (None, "a6_solve_27b"):
        # a6 at the 27B shape: d = 5120, 48 maps, sums over 16,384 rows accumulated on the device
        c = synth.DENSE27B
        out["a6_solve_27b"] = _solve_row(dev, c.d, c.d, c.P, c.calib_n, c.lam, c.index, flags, peak_tflops,
                                         f"27b-shaped ridge solve, d={c.d}, {c.P} maps, lambda={c.lam}, "
                                         f"sums from {c.calib_n} calibration rows")

    if only in (None, "a6_solve_xmodel"):
        # a6 for the cross-model mapper: 8192 concatenated features -> 1024 target columns, one map
        # (one kind of one target layer), sums over 131,072 rows
        x = synth.XMODEL
        out["a6_solve_xmodel"] = _solve_row(dev, x.d_in, x.KV, 1, x.calib_n, x.lam, x.index, flags, peak_tflops,
                                            f"cross-model ridge solve, d_in={x.d_in} -> d_out={x.KV}, one map, "
                                            f"lambda={x.lam}, sums from {x.calib_n} rows")

    if only in (None, "a7_xmodel"):
        # a7: cross-model mapper, 40 -> 64 layers, k = 8, 8 x 128 heads, N = 32768
        x = synth.XMODEL
        if capture:
            x = dataclasses.replace(x, name="xmodel 12->4 layers 8x128 k8 N32768 (capture size)", L_src=12, L_tgt=4)
        inp = synth.xmodel_inputs(x, device=dev)
        xd = rf.rf_xmodel_desc(L_src=x.L_src, L_tgt=x.L_tgt, k=x.k, n_kv_heads=x.H, head_dim=x.hd, N=x.N,
                               theta_src=x.theta_src, theta_tgt=x.theta_tgt, pos_offset=0, flags=flags)
        kt = torch.empty((x.L_tgt, x.N, x.KV), dtype=torch.bfloat16, device=dev)
        vt = torch.empty_like(kt)
        wsb = rf.rf_xmodel_workspace_bytes(xd)
        ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
        src = torch.as_tensor(inp["src"], dtype=torch.int32, device=dev)
        ms, stages = _timed(lambda: rf.rf_xmodel_map(xd, src, inp["k_src"], inp["v_src"], inp["Wk"], inp["bk"],
                                                     inp["Wv"], inp["bv"], kt, vt, None, ws, wsb), 3, stream)
        flops = 2.0 * x.N * x.d_in * 2 * x.KV * x.L_tgt
        gm = stages.get("xmodel_gemm", ms)
        out["a7_xmodel"] = {"workload": x.name, "ms_per_call": ms, "tflops": flops / (ms / 1e3) / 1e12,
                            "gemm_ms": gm, "gemm_frac_of_bf16_peak": flops / (gm / 1e3) / 1e12 / peak_tflops,
                            "stages_ms": stages,
                            "pages_context": "277.6 ms for a 40->64 layer pair at 32K on unstated hardware (context only)"}
        del inp, kt, vt, ws
        torch.cuda.empty_cache()

    if only in (None, "next3_map_storage_8b"):
        # Map storage at the bench workload (8B shape): the resident fill against the
        # layer-by-layer fill with maps on the device or the host, bf16 or int8
        c = synth.LLAMA8B
        inp = synth.fill_inputs(c, device=dev)
        fd, Wk, Wv = _prefolded(c, inp, flags)
        q = torch.empty((c.P, c.d, c.d), dtype=torch.int8, device=dev)
        qs = torch.empty((c.P, c.d), dtype=torch.float32, device=dev)
        rf.rf_quantize_maps_int8(fd, inp["A"], q, qs)
        A_host = inp["A"].cpu().pin_memory()
        q_host = q.cpu().pin_memory()
        kc = torch.zeros((c.L, c.N, c.KV), dtype=torch.bfloat16, device=dev)
        vc = torch.zeros_like(kc)
        nf = torch.zeros(1, dtype=torch.int32, device=dev)
        row = {"workload": workload_label(c), "map_bytes_bf16": c.P * c.d * c.d * 2, "map_bytes_int8": c.P * c.d * c.d}
        wsb = rf.rf_fill_workspace_bytes(fd)
        ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
        row["resident_ms"], _ = _timed(lambda: rf.rf_fill_kv(fd, inp["x_S"], c.d, inp["mask"], inp["A"], inp["b"], None,
                                                             Wk, Wv, kc, vc, c.N * c.KV, c.KV, nf, None, ws, wsb), 3,
                                       stream)
        row["resident_workspace_bytes"] = wsb
        del ws
        variants = {"layered_device_bf16": rf.map_source(rf.RF_MAPS_BF16, inp["A"]),
                    "layered_host_bf16": rf.map_source(rf.RF_MAPS_BF16, A_host, on_host=True),
                    "layered_device_int8": rf.map_source(rf.RF_MAPS_INT8, q, row_scale=qs),
                    "layered_host_int8": rf.map_source(rf.RF_MAPS_INT8, q_host, on_host=True, row_scale=qs)}
        for key, ms_ in variants.items():
            wsb = rf.rf_fill_layered_workspace_bytes(fd, ms_)
            ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
            row[f"{key}_ms"], st = _timed(lambda: rf.rf_fill_kv_layered(fd, inp["x_S"], c.d, inp["mask"], ms_, inp["b"],
                                                                        None, Wk, Wv, kc, vc, c.N * c.KV, c.KV, nf,
                                                                        None, ws, wsb), 3, stream)
            row[f"{key}_workspace_bytes"] = wsb
            if "int8_expand" in st:
                row[f"{key}_expand_ms"] = st["int8_expand"]
            del ws
        out["next3_map_storage_8b"] = row
        del inp, kc, vc, Wk, Wv, q, qs, A_host, q_host
        torch.cuda.empty_cache()

    if only in (None, "next3_map_storage_27b"):
        # The 27B deployment's map storage: the 48 maps in int8 (1.26 GB, the pages'
        # "1.2 GiB") streamed layer by layer from pinned host memory, against the same
        # int8 maps on the device, the layered fill from the bf16 maps on the device,
        # and the resident bf16 fill. The synthetic maps are I + N(0, 0.02²/d): their
        # per-row int8 codes are 0 off the diagonal for almost every entry, so the int8
        # arms multiply mostly zeros, draw less power and run at higher power-capped
        # clocks; compare the int8 arms with each other (the cost of streaming) and the
        # bf16 arms with each other (the cost of going layer by layer).
        c = synth.DENSE27B
        inp = synth.fill_inputs(c, device=dev)
        fd, Wk, Wv = _prefolded(c, inp, flags)
        q = torch.empty((c.P, c.d, c.d), dtype=torch.int8, device=dev)
        qs = torch.empty((c.P, c.d), dtype=torch.float32, device=dev)
        rf.rf_quantize_maps_int8(fd, inp["A"], q, qs)
        q_host = q.cpu().pin_memory()
        kc = torch.zeros((c.P, c.N, c.KV), dtype=torch.bfloat16, device=dev)
        vc = torch.zeros_like(kc)
        nf = torch.zeros(1, dtype=torch.int32, device=dev)
        fd0 = rf.rf_fill_desc(d=c.d, d_in=c.d_in, L=c.P, S=0, N=c.N, T=c.T, n_kv_heads=c.H, head_dim=c.hd,
                              rope_theta=c.rope_theta, rms_eps=c.rms_eps, pos_offset=c.pos_offset, flags=fd.flags)
        row = {"workload": workload_label(c), "map_bytes_bf16": c.P * c.d * c.d * 2, "map_bytes_int8": c.P * c.d * c.d}
        wsb = rf.rf_fill_workspace_bytes(fd0)
        ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
        row["resident_bf16_ms"], _ = _timed(lambda: rf.rf_fill_kv(fd0, inp["x_S"], c.d, inp["mask"], inp["A"],
                                                                  inp["b"], None, Wk, Wv, kc, vc, c.N * c.KV, c.KV, nf,
                                                                  None, ws, wsb), 3, stream)
        row["resident_workspace_bytes"] = wsb
        del ws
        torch.cuda.empty_cache()
        for key, ms_ in (("layered_device_bf16", rf.map_source(rf.RF_MAPS_BF16, inp["A"])),
                         ("layered_device_int8", rf.map_source(rf.RF_MAPS_INT8, q, row_scale=qs)),
                         ("layered_host_int8", rf.map_source(rf.RF_MAPS_INT8, q_host, on_host=True, row_scale=qs))):
            wsb = rf.rf_fill_layered_workspace_bytes(fd0, ms_)
            ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
            row[f"{key}_ms"], st = _timed(lambda: rf.rf_fill_kv_layered(fd0, inp["x_S"], c.d, inp["mask"], ms_,
                                                                        inp["b"], None, Wk, Wv, kc, vc, c.N * c.KV,
                                                                        c.KV, nf, None, ws, wsb), 3, stream)
            row[f"{key}_workspace_bytes"] = wsb
            if "int8_expand" in st:
                row[f"{key}_expand_ms"] = st["int8_expand"]
            del ws
        row["note"] = ("int8 codes of the synthetic maps are mostly 0 off the diagonal: the int8 arms draw less "
                       "power and clock higher; compare int8 with int8 and bf16 with bf16")
        out["next3_map_storage_27b"] = row
        del inp, kc, vc, Wk, Wv, q, qs, q_host
        torch.cuda.empty_cache()

    if only in (None, "next2_key_norm_qwen3"):
        # Key normalisation: the Qwen3-8B-shaped fill without and with per-head K norm
        c = synth.QWEN3_8B
        inp = synth.fill_inputs(c, device=dev)
        kg = synth.key_norm_gain(c, device=dev)
        fd, Wk, Wv = _prefolded(c, inp, flags)
        kc = torch.zeros((c.L, c.N, c.KV), dtype=torch.bfloat16, device=dev)
        vc = torch.zeros_like(kc)
        wsb = rf.rf_fill_workspace_bytes(fd)
        ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
        nf = torch.zeros(1, dtype=torch.int32, device=dev)
        row = {"workload": f"qwen3-8b-shaped fill (d={c.d}, {c.P} upper layers, N={c.N}, T={c.T}, no exact rows)"}
        for key, gain_ptr in (("plain", None), ("key_norm", kg.data_ptr())):
            fd.k_norm_gain = gain_ptr
            ms, st = _timed(lambda: rf.rf_fill_kv(fd, inp["x_S"], c.d, inp["mask"], inp["A"], inp["b"], None, Wk, Wv, kc,
                                                  vc, c.N * c.KV, c.KV, nf, None, ws, wsb), 5, stream)
            n_fill = int(nf.item())
            f_flops = 2.0 * n_fill * c.P * (c.d * c.d + c.d * 2 * c.KV)
            row[f"{key}_ms"] = ms
            row[f"{key}_tflops"] = f_flops / (ms / 1e3) / 1e12
            row[f"{key}_kv_gemm_ms"] = st.get("kv_gemm")
            row[f"{key}_map_gemm_ms"] = st.get("map_gemm")
        out["next2_key_norm_qwen3"] = row
        del inp, kc, vc, ws, Wk, Wv
        torch.cuda.empty_cache()

    if only in (None, "next4_nonsquare_flash_next"):
        # Non-square maps: the Flash-Next-shaped fill (10,240 -> 2,560, 24 upper layers)
        c = synth.FLASH_NEXT
        inp = synth.fill_inputs(c, device=dev)
        fd, Wk, Wv = _prefolded(c, inp, flags)
        kc = torch.zeros((c.L, c.N, c.KV), dtype=torch.bfloat16, device=dev)
        vc = torch.zeros_like(kc)
        wsb = rf.rf_fill_workspace_bytes(fd)
        ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
        nf = torch.zeros(1, dtype=torch.int32, device=dev)
        ms, st = _timed(lambda: rf.rf_fill_kv(fd, inp["x_S"], c.d_in, inp["mask"], inp["A"], inp["b"], None, Wk, Wv, kc,
                                              vc, c.N * c.KV, c.KV, nf, None, ws, wsb), 3, stream)
        n_fill = int(nf.item())
        f_flops = 2.0 * n_fill * c.P * (c.d * c.d_in + c.d * 2 * c.KV)
        mg = st.get("map_gemm")
        out["next4_nonsquare_flash_next"] = {
            "workload": c.name + f", n_fill={n_fill}", "fill_ms": ms, "fill_tflops": f_flops / (ms / 1e3) / 1e12,
            "fill_frac_of_bf16_peak": f_flops / (ms / 1e3) / 1e12 / peak_tflops,
            "map_gemm_ms": mg, "map_gemm_tflops": 2.0 * n_fill * c.P * c.d * c.d_in / (mg / 1e3) / 1e12 if mg else None,
            "fill_row_layers_per_s": n_fill * c.P / (ms / 1e3), "stages_ms": st}
        del inp, kc, vc, ws, Wk, Wv
        torch.cuda.empty_cache()

    if only in (None, "next1_value_rescale_27b"):
        # Value rescale (the 27B deployment, c = 512), then the 27B fill with the scale
        c = synth.DENSE27B
        n_tail = 512
        inp = synth.fill_inputs(c, device=dev)
        x_exact = synth.rescale_inputs(c, inp["x_S"], n_tail, device=dev)
        fd, Wk, Wv = _prefolded(c, inp, flags)
        vs = torch.empty((c.P, c.H), dtype=torch.float32, device=dev)
        wsb = rf.rf_value_scale_workspace_bytes(fd, n_tail)
        ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
        ms_scale, st_scale = _timed(lambda: rf.rf_value_scale(fd, n_tail, inp["x_S"], c.d, x_exact, c.d, inp["A"], inp["b"],
                                                              None, Wv, vs, None, ws, wsb), 3, stream)
        del ws
        fd.v_scale = vs.data_ptr()
        kc = torch.zeros((c.L, c.N, c.KV), dtype=torch.bfloat16, device=dev)
        vc = torch.zeros_like(kc)
        wsb = rf.rf_fill_workspace_bytes(fd)
        ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
        nf = torch.zeros(1, dtype=torch.int32, device=dev)
        ms_fill, st_fill = _timed(lambda: rf.rf_fill_kv(fd, inp["x_S"], c.d, inp["mask"], inp["A"], inp["b"], None, Wk, Wv,
                                                        kc, vc, c.N * c.KV, c.KV, nf, None, ws, wsb), 3, stream)
        n_fill = int(nf.item())
        f_flops = 2.0 * n_fill * c.P * (c.d * c.d + c.d * 2 * c.KV)
        s_flops = 2.0 * n_tail * c.P * (c.d * c.d + 2 * c.d * c.KV)
        out["next1_value_rescale_27b"] = {
            "workload": f"27b-shaped deployment: value rescale over c={n_tail} tail rows, then the fill with the scale "
                        f"(d={c.d}, {c.P} upper layers, n_fill={n_fill})",
            "rescale_ms": ms_scale, "rescale_tflops": s_flops / (ms_scale / 1e3) / 1e12, "rescale_stages_ms": st_scale,
            "fill_ms": ms_fill, "fill_tflops": f_flops / (ms_fill / 1e3) / 1e12,
            "fill_frac_of_bf16_peak": f_flops / (ms_fill / 1e3) / 1e12 / peak_tflops,
            "fill_row_layers_per_s": n_fill * c.P / (ms_fill / 1e3), "fill_stages_ms": st_fill}
        del inp, kc, vc, ws, Wk, Wv, vs, x_exact
        torch.cuda.empty_cache()

    if only in (None, "next4a_source_selection_xmodel"):
        out["next4a_source_selection_xmodel"] = run_selection(dev, peak_tflops, flags)

    return out


def _solve_row(dev, d_in, d_out, P, n, lam, index, flags, peak_tflops, label):
    """One rf_solve row: planted calibration rows accumulated on the device, then the
    solve timed unrefined and with one refinement sweep."""
    import torch

    import ridge_map_kv_gb300 as rf
    import synth
    stream = torch.cuda.current_stream(dev)
    st = _zero_stats(d_in, d_out, P, dev)
    cs = rf.calib_stats_struct(st["G"], st["C"], st["sx"], st["sy"], st["n"])
    cd = rf.rf_calib_desc(d_in=d_in, d_out=d_out, n_maps=P, flags=flags)
    chunk = min(n, 16384)
    for r0 in range(0, n, chunk):      # rows generated in chunks outside the timed calls
        cal = synth.calib_inputs(d_in, d_out, P, chunk, index=index, device=dev, salt=r0 // chunk)
        rf.rf_calib_accumulate(cd, cal["X"], d_in, cal["Y"], d_out, chunk * d_out, chunk, cs)
        del cal
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    A = torch.empty((P, d_out, d_in), dtype=torch.float32, device=dev)
    b = torch.empty((P, d_out), dtype=torch.float32, device=dev)
    Ab = torch.empty((P, d_out, d_in), dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    wsb = rf.rf_solve_workspace_bytes(cd)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    row = {"workload": label, "workspace_bytes": wsb}
    for refine in (0, 1):
        ms, stages = _timed(lambda: rf.rf_solve(cd, cs, lam, rf.RF_ALPHA_TRACE, refine, A, b, Ab, None, status, ws,
                                                wsb), 1, stream)
        row[f"refine_{refine}_ms"] = ms
        row[f"refine_{refine}_stages_ms"] = stages
    assert int(status.item()) == 0
    # A_p = Cc_pᵀ H^-1: 2 P d_out d_in² fp32-accurate flops, as six bf16 plane products
    prod = 2.0 * P * d_out * d_in ** 2
    pm = row["refine_0_stages_ms"].get("solve_product")
    if pm:
        row["product_fp32_tflops"] = prod / (pm / 1e3) / 1e12
        row["product_bf16_plane_tflops"] = 6.0 * prod / (pm / 1e3) / 1e12
        row["product_frac_of_bf16_peak"] = row["product_bf16_plane_tflops"] / peak_tflops
    # factorisation and inverse: Cholesky d³/3, L^-1 d³/3, H^-1 = L^-ᵀL^-1 d³ (fp32-equivalent)
    fm = row["refine_0_stages_ms"].get("solve")
    if fm:
        row["factor_inverse_fp32_tflops"] = (5.0 / 3.0) * d_in ** 3 / (fm / 1e3) / 1e12
    rm = row["refine_1_stages_ms"].get("solve_refine")
    if rm:
        # one sweep = the residual A_p H plus the correction R_p H^-1 (see a6_solve)
        row["refine_sweep_ms"] = rm
        row["refine_product_equiv_tflops"] = 2.0 * prod / (rm / 1e3) / 1e12
    row["solve_fp32_equiv_tflops_unrefined"] = (prod + (5.0 / 3.0) * d_in ** 3) / (row["refine_0_ms"] / 1e3) / 1e12
    del st, cs, A, b, Ab, ws
    torch.cuda.empty_cache()
    return row


def run_selection(dev, peak_tflops, flags=0, n_targets=0, n_sources=0):
    """Greedy source-layer selection for the 40 -> 64 layer pair (8 x 128 heads,
    k = 8, keys and values scored jointly): the calibration sums over all 40
    source layers (40,960 features) from 131,072 rows, then rf_select_sources.
    Rows are generated in chunks outside the timed calls."""
    import torch

    import ridge_map_kv_gb300 as rf
    import synth
    stream = torch.cuda.current_stream(dev)
    cfg = synth.SELECT_XMODEL
    if n_sources > 0:
        cfg = dataclasses.replace(cfg, L_src=max(cfg.k, n_sources))
    T = cfg.L_tgt if n_targets <= 0 else min(n_targets, cfg.L_tgt)
    D, F, chunk = cfg.D, cfg.F, 16384
    cd = rf.rf_calib_desc(d_in=D, d_out=F, n_maps=T, flags=flags)
    stats, calib_ms = [], []
    for kind in (0, 1):
        ld = synth.selection_loadings(cfg, kind, dev)
        st = {"G": torch.zeros((D, D), dtype=torch.float64, device=dev),
              "C": torch.zeros((T, D, F), dtype=torch.float64, device=dev),
              "sx": torch.zeros(D, dtype=torch.float64, device=dev),
              "sy": torch.zeros((T, F), dtype=torch.float64, device=dev),
              "syy": torch.zeros((T, F), dtype=torch.float64, device=dev),
              "n": torch.zeros(1, dtype=torch.int64, device=dev)}
        cs = rf.calib_stats_struct(st["G"], st["C"], st["sx"], st["sy"], st["n"], st["syy"])
        total = 0.0
        for ch in range(cfg.n // chunk):
            r = synth.selection_rows(cfg, kind, chunk, ch, dev, ld)
            Y = r["Y"][:T].contiguous()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record(stream)
            rf.rf_calib_accumulate(cd, r["X"], D, Y, F, chunk * F, chunk, cs)
            e1.record(stream)
            torch.cuda.synchronize()
            total += e0.elapsed_time(e1)
            del r, Y
        stats.append((st, cs))
        calib_ms.append(total)
        del ld
    torch.cuda.empty_cache()
    d = rf.rf_select_desc(L_src=cfg.L_src, F=F, n_targets=T, d_out=F, head_dim=cfg.hd, k=cfg.k, n_kinds=2,
                          group=min(8, T), flags=flags)
    wsb = rf.rf_select_workspace_bytes(d)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    sel = torch.empty((T, cfg.k), dtype=torch.int32, device=dev)
    r2 = torch.empty((2, T, cfg.k, cfg.L_src), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ms, stages = _timed(lambda: rf.rf_select_sources(d, [cs for _, cs in stats], cfg.lam, rf.RF_ALPHA_TRACE, sel, r2,
                                                     status, ws, wsb), 1, stream)
    assert int(status.item()) == 0
    # fp32-accurate products (each is six bf16 plane products on the tensor cores):
    # per pass of Q problems and step j (m = jF features chosen), the scores of the
    # L_src - j candidates left (2 D F Ft over those layers), and for j < k-1 z_b
    # (2 Ft F²) and, over the L_src - j - 1 layers left once b is chosen, the new
    # factor column (2 D F m + 2 D F²) and the Schur-block and cross-term updates
    # (2 D F² + 2 Ft F D); the chosen layers' units run nothing. The scores, z_b and
    # the new column's "× L_b^-ᵀ" multiply by a lower-triangular L^-1: algorithmically
    # (F+1)/2F of a full product, and the kernel runs the tiles up to each column
    # tile's diagonal, (T+1)/2T with T = F/256.
    n_prob = 2 * T
    L = cfg.L_src
    tri_alg, tri_exec = (F + 1) / (2.0 * F), (F // 256 + 1) / (2.0 * (F // 256))
    prod, prod_exec = 0.0, 0.0
    for j in range(cfg.k):
        m = j * F
        left, after = (L - j) / L, (L - j - 1) / L
        full = (2.0 * D * F * m + 2.0 * D * F * F + 2.0 * F * F * D) * after if j < cfg.k - 1 else 0.0
        tri = 2.0 * D * F * F * left + ((2.0 * D * F * F * after + 2.0 * F * F * F) if j < cfg.k - 1 else 0.0)
        prod += full + tri_alg * tri
        prod_exec += full + tri_exec * tri
    prod *= n_prob
    prod_exec *= n_prob
    gm = stages.get("select_gemm", ms)
    # fp32 SIMT factorisation of every candidate's F x F Schur block at every step
    # (Cholesky F³/3 and triangular inverse F³/3, algorithmic)
    fact = n_prob * cfg.L_src * cfg.k * (2.0 * F ** 3 / 3.0)
    sustained = measured_peaks().get("bf16_tflops_sustained") or peak_tflops   # seconds-long timed region
    fm = stages.get("select_factor", ms)
    cflops = 1.0 * cfg.n * D * (D + 1) + 2.0 * cfg.n * D * F * T
    return {
        "workload": f"{cfg.name}: source selection for {T} target layers, keys and values jointly, "
                    f"calibration sums over all {cfg.L_src} source layers ({D} features) from {cfg.n} rows",
        "calibration_ms_per_kind": calib_ms,
        "calibration_tflops": cflops / (sum(calib_ms) / 2 / 1e3) / 1e12,
        "select_ms": ms, "select_stages_ms": stages,
        "select_products_fp32_tflops": prod / (gm / 1e3) / 1e12,
        "select_products_algorithmic_fp32_tflop": prod / 1e12,
        "select_products_executed_fp32_tflop": prod_exec / 1e12,
        "select_products_bf16_plane_tflops": 6.0 * prod_exec / (gm / 1e3) / 1e12,
        "select_products_frac_of_sustained_bf16_peak": 6.0 * prod_exec / (gm / 1e3) / 1e12 / sustained,
        "select_factor_fp32_tflops": fact / (fm / 1e3) / 1e12,
        "select_workspace_bytes": wsb,
        "first_target_layers": sel[0].tolist(),
        "pages_context": "47-87 min to fit one pair's mapper on 8 H100s (XᵀX dominant; whole fit, context only)"}


# --------------------------------------------------------------------------- #
# Reference arm: the fp64 oracle on the host cores
# --------------------------------------------------------------------------- #
def run_reference(args):
    """The reference arm: the fp64 oracle as it stands, on the host cores, over the
    same workload, metric and unit as our arm. Each step is a bounded sample of the
    workload (REF_ROWS_PER_STEP filled rows x every upper layer), so that K steps end
    within a few minutes."""
    import synth
    ws_n, rank, _ = dist_env()
    if rank != 0:
        return
    cfg = workloads()[args.workload]
    inp = synth.fill_inputs(cfg, device="cpu")
    n_fill, units = fill_units(cfg, inp["mask"])
    rows_per_step = REF_ROWS_PER_STEP
    oi = OracleInputs(cfg, inp)
    del inp
    for _ in range(max(args.warmup, 3)):
        cpu_oracle_rate(oi, 2, seed=0)
    t = 0.0
    done = 0
    cores = host_cores()
    for k in range(args.steps):
        _, dt, n, cores = cpu_oracle_rate(oi, rows_per_step, seed=100 + k)
        t += dt
        done += n * cfg.P
    value = done / t
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws_n,
            "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": 1e3 * t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": workload_label(cfg), "n_fill": n_fill,
                       "upper_layers": cfg.P, "sample_rows_per_step": rows_per_step},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"{rows_per_step} filled rows x {cfg.P} upper layers per step"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


REF_ROWS_PER_STEP = 16


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    elif args.selection_only:
        run_selection_only(args)
    elif args.extra:
        run_extra_only(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
