#!/usr/bin/env python3
"""Benchmark of the PlaneZip block codec on GB300: raw-byte GB/s of compress
and decompress through the C ABI, the compression ratio, and the roofline
fraction of the dominant kernel, on the 1 GiB throughput sweep.

One step = every segment of the sweep compressed (one pz_compress call per
segment) and then decompressed (one pz_decompress call per segment), back to
back on one stream, inputs resident in HBM. Each segment (128-256 MiB) is
larger than the 129 MB L2, so no flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With N > 1 (launched by torch.distributed.run) every rank runs an
independent replica on its own GPU (the codec has no exchange step); the
step time is the maximum over ranks and `value` counts all ranks' bytes.
`--impl reference` times the CPU oracle (the only reference this codec has),
chunk-parallel over all host cores, on a bounded sample of the same workload,
on rank 0 only.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

METRIC = "raw-byte GB/s compress & decompress (BF16/FP32) vs HBM roofline; ratio"
FALLBACK_HBM_GBS = 6800.0
WORKLOAD = ("1 GiB throughput sweep: {ReLU, smooth conv, causal attention} x {FP32, BF16} "
            "at 128 MiB each + 256 MiB uniform u32; one compress call per segment, then all "
            "segments decompressed, back to back on one stream")

# DRAM bytes (read + write) per encoder launch on the 1 GiB sweep: the mean
# over its seven segments of dram__bytes_read.sum + dram__bytes_write.sum, one
# ncu capture of the encoder per segment workload. The counters describe the
# encoder as compiled from the device sources whose sha256 is recorded with
# them: once those sources change, `roofline.traffic` is reported as null
# until the encoder is captured again. It is also null when the sweep's
# dominant call is not the encoder.
NCU_ENCODER_TRAFFIC = {
    "sources": ("lossless_bit_plane_gb300/csrc/encode.cu", "lossless_bit_plane_gb300/csrc/pz_encode_block.cuh",
                "lossless_bit_plane_gb300/csrc/pz_device.cuh", "lossless_bit_plane_gb300/csrc/pz_format.cuh"),
    "sources_sha256": "feb1ff2022f50378dd0c2bf177dbdb239c9568f245c57fe9573d33004610aa26",
    "bytes_per_launch": 211.54e6,
}


def encoder_traffic():
    """The recorded ncu DRAM bytes per encoder launch, or None if the
    encoder's device sources are not the ones they were measured on."""
    import hashlib

    h = hashlib.sha256()
    for f in NCU_ENCODER_TRAFFIC["sources"]:
        h.update((ROOT / f).read_bytes())
    return NCU_ENCODER_TRAFFIC["bytes_per_launch"] if h.hexdigest() == NCU_ENCODER_TRAFFIC["sources_sha256"] else None


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-sample-mib", type=float, default=4.0,
                    help="MiB per segment timed through the CPU oracle")
    ap.add_argument("--cpu-parallel-mib", type=float, default=16.0,
                    help="MiB per segment timed through the CPU oracle chunk-parallel over all host cores (0: skip)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the sizes-only, ablation and swap sections (run after the timed region)")
    ap.add_argument("--seg-mib", type=int, default=128,
                    help="segment size in MiB for a single-segment workload (<kind>_<dtype>; attention wants a "
                         "multiple of 4 MiB for FP32 and 2 MiB for BF16); small profiling cases")
    ap.add_argument("--workload", default="sweep",
                    help="'sweep' (the 1 GiB sweep, the headline), a parity config (config1, config2, config3, "
                         "config4_fp32, config4_bf16), or one sweep segment as <kind>_<dtype>, e.g. "
                         "attention_fp32, conv_bf16, random_u32 (used for small profiling cases)")
    return ap.parse_args()


# ------------------------------------------------------------- distributed

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def init_dist(world: int, backend: str):
    import torch.distributed as dist

    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, value: float, device=None) -> float:
    if dist is None:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples every 200 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

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
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------- workload

def make_workload(name: str = "sweep", seg_mib: int = 128):
    from lossless_bit_plane_gb300 import workloads as W

    if name == "sweep":
        return W.sweep_1gib()
    configs = {"config1": lambda: [W.relu_fp32_4mib()], "config2": lambda: [W.conv_bf16()],
               "config3": lambda: [W.attention_bf16()], "config4_fp32": lambda: W.mlp_ln(dtype="fp32"),
               "config4_bf16": lambda: W.mlp_ln(dtype="bf16")}
    if name in configs:
        return configs[name]()
    kind, dtype = name.rsplit("_", 1)
    return [W.sweep_segment(kind, dtype, seg_bytes=seg_mib << 20)]


CONFIG_LABELS = {
    "config1": "FP32 post-ReLU tensor, 1,048,576 elements (4 MiB), seed 0",
    "config2": "BF16 conv feature map [32,64,56,56], blurred ReLU fields, seed 1",
    "config3": "BF16 causal attention probabilities [8,12,1024,1024] (192 MiB), seed 2",
    "config4_fp32": "FP32 GELU [8,1024,3072] + LayerNorm [8,1024,768] outputs, seed 3",
    "config4_bf16": "BF16 GELU [8,1024,3072] + LayerNorm [8,1024,768] outputs, seed 3",
}


def workload_label(name: str) -> str:
    if name == "sweep":
        return WORKLOAD
    return CONFIG_LABELS.get(name, f"one 1 GiB-sweep segment distribution: {name}")


def peak_hbm():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        try:
            return float(json.loads(p.read_text())["hbm_gbs"]), "measured"
        except (KeyError, ValueError):
            pass
    return FALLBACK_HBM_GBS, "fallback"


# -------------------------------------------------------------- CPU oracle

def cpu_oracle_sample(segs, mib: float):
    """Round trip of the first `mib` MiB of every segment through the oracle
    (single thread); returns (raw bytes, compress s, decompress s)."""
    import oracle

    oracle.build()
    nb, tc, td = 0, 0.0, 0.0
    for t in segs:
        n = min(t.nbytes, int(mib * (1 << 20)))
        piece = t.data[:n]
        t0 = time.perf_counter()
        s = oracle.compress(piece, t.elem_width)
        t1 = time.perf_counter()
        back = oracle.decompress(s, n, t.elem_width)
        t2 = time.perf_counter()
        assert back == piece.tobytes()
        nb += n
        tc += t1 - t0
        td += t2 - t1
    return nb, tc, td


def cpu_oracle_parallel(segs, mib: float):
    """The same oracle calls, chunk-parallel over the host's cores: the first
    `mib` MiB of every segment is cut at chunk boundaries into one slice per
    thread, and each thread round-trips its slice (chunks are coded on their
    own, so the slices' streams concatenate, size tables first, into the
    whole sample's stream). The oracle's C calls run without the GIL.
    Returns (raw bytes, compress s, decompress s, threads)."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle

    oracle.build()
    threads = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    nb, tc, td = 0, 0.0, 0.0
    with ThreadPoolExecutor(max_workers=threads) as pool:
        for t in segs:
            n = min(t.nbytes, int(mib * (1 << 20)))
            raw = t.data[:n].view(np.uint8)
            C = (n + 4095) // 4096
            cuts = [4096 * (C * i // threads) for i in range(threads + 1)]
            slices = [raw[a:min(n, b)] for a, b in zip(cuts[:-1], cuts[1:]) if a < min(n, b)]
            t0 = time.perf_counter()
            streams = list(pool.map(lambda p: oracle.compress(p, t.elem_width), slices))
            t1 = time.perf_counter()
            backs = list(pool.map(lambda sp: oracle.decompress(sp[0], sp[1].size, t.elem_width),
                                  zip(streams, slices)))
            t2 = time.perf_counter()
            assert b"".join(backs) == raw.tobytes()
            nb += n
            tc += t1 - t0
            td += t2 - t1
    return nb, tc, td, threads


def run_reference(args, rank: int):
    """The reference arm: the oracle, chunk-parallel over all host cores, on a
    bounded sample of the workload per step (rank 0 only)."""
    if rank != 0:
        return 0
    segs = make_workload(args.workload, args.seg_mib)
    mib = min(args.cpu_parallel_mib, 4.0) if args.cpu_parallel_mib > 0 else 1.0
    for _ in range(args.warmup):
        cpu_oracle_parallel(segs, mib)
    nb_tot, tc_tot, td_tot, threads = 0, 0.0, 0.0, 1
    for _ in range(args.steps):
        nb, tc, td, threads = cpu_oracle_parallel(segs, mib)
        nb_tot += nb
        tc_tot += tc
        td_tot += td
    value = nb_tot / (tc_tot + td_tot) / 1e9
    sample = (f"first {mib:g} MiB of each of the {len(segs)} segments of the workload per step, cut at chunk "
              f"boundaries into one slice per thread, compress + decompress")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * (tc_tot + td_tot) / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u32",
        "data": "synthetic", "config": {"workload": workload_label(args.workload), "sample": sample},
        "compress_gbs": nb_tot / tc_tot / 1e9, "decompress_gbs": nb_tot / td_tot / 1e9,
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# -------------------------------------------------------------------- GPU

def run_ours(args, rank: int, world: int, local: int):
    import torch

    from lossless_bit_plane_gb300 import _lib, build

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    build.build()
    _lib.load()

    segs = make_workload(args.workload, args.seg_mib)
    stream = torch.cuda.current_stream(dev)
    d_in = [torch.from_numpy(t.data).to(dev) for t in segs]
    d_out = [torch.empty(_lib.pz_max_compressed_bytes(t.nbytes), dtype=torch.uint8, device=dev) for t in segs]
    d_tot = torch.zeros(len(segs), dtype=torch.int64, device=dev)
    d_back = [torch.empty(t.nbytes, dtype=torch.uint8, device=dev) for t in segs]
    d_st = torch.zeros(len(segs), dtype=torch.int32, device=dev)
    sh = stream.cuda_stream

    # workloads with a segment smaller than 128 MiB would run out of L2: every
    # timed call is then preceded by a 256 MiB write outside its events
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if min(t.nbytes for t in segs) < (128 << 20) \
        else None

    def flush():
        if flush_buf is not None:
            flush_buf.fill_(1)

    def compress_all(evs=None):
        for i, t in enumerate(segs):
            if evs:
                flush()
                evs[i][0].record(stream)
            rc = _lib.pz_compress(d_in[i].data_ptr(), t.nbytes, t.elem_width, d_out[i].data_ptr(), d_out[i].numel(),
                                  d_tot[i:i + 1].data_ptr(), sh)
            assert rc == 0, rc
            if evs:
                evs[i][1].record(stream)

    totals_host = None

    def decompress_all(totals, evs=None):
        for i, t in enumerate(segs):
            if evs:
                flush()
                evs[i][0].record(stream)
            rc = _lib.pz_decompress(d_out[i].data_ptr(), int(totals[i]), t.elem_width, d_back[i].data_ptr(), t.nbytes,
                                    d_st[i:i + 1].data_ptr(), sh)
            assert rc == 0, rc
            if evs:
                evs[i][1].record(stream)

    # first pass: totals (the decompressor's comp_bytes) and a correctness check
    compress_all()
    torch.cuda.synchronize()
    totals_host = d_tot.cpu().tolist()
    decompress_all(totals_host)
    torch.cuda.synchronize()
    assert d_st.cpu().tolist() == [0] * len(segs)
    for i in range(len(segs)):
        assert torch.equal(d_back[i], d_in[i]), f"round trip failed on segment {i}"

    for _ in range(args.warmup):
        compress_all()
        decompress_all(totals_host)
    torch.cuda.synchronize()

    nseg = len(segs)
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    c_evs = [[[ev(), ev()] for _ in range(nseg)] for _ in range(args.steps)]
    d_evs = [[[ev(), ev()] for _ in range(nseg)] for _ in range(args.steps)]
    start, stop = ev(), ev()
    clocks = ClockSampler(local) if rank == 0 else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    barrier(dist)
    torch.cuda.synchronize()
    start.record(stream)
    for k in range(args.steps):
        compress_all(c_evs[k])
        decompress_all(totals_host, d_evs[k])
    stop.record(stream)
    torch.cuda.synchronize()
    barrier(dist)
    clk = clocks.stop() if clocks else None
    elapsed_ms = start.elapsed_time(stop)
    elapsed_ms = max_over_ranks(dist, elapsed_ms, dev)

    totals_now = d_tot.cpu().tolist()
    assert totals_now == totals_host
    launches_per_step = count_launches(lambda: (compress_all(), decompress_all(totals_host)))
    raw = sum(t.nbytes for t in segs)
    comp = sum(totals_host)
    t_c = [sum(c_evs[k][i][0].elapsed_time(c_evs[k][i][1]) for k in range(args.steps)) / args.steps for i in range(nseg)]
    t_d = [sum(d_evs[k][i][0].elapsed_time(d_evs[k][i][1]) for k in range(args.steps)) / args.steps for i in range(nseg)]
    tc_ms, td_ms = sum(t_c), sum(t_d)
    peak, peak_kind = peak_hbm()
    # algorithmic bytes per call: raw read + stream written (compress),
    # stream read + raw written (decompress); both are raw + stream
    alg = [t.nbytes + totals_host[i] for i, t in enumerate(segs)]
    comp_ach = sum(alg) / (tc_ms * 1e-3) / 1e9
    dec_ach = sum(alg) / (td_ms * 1e-3) / 1e9
    dominant = "pz_encode" if tc_ms >= td_ms else "pz_decode"
    ach = comp_ach if dominant == "pz_encode" else dec_ach

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, segs, d_out, d_back, d_tot, d_st, totals_host, dev, stream, world, dist)
    sizes = {"size_only": None, "ablation": None} if args.no_extras else run_sizes(args, segs, d_in, totals_host, dev,
                                                                                      stream)
    swap = None if args.no_extras else run_swap(segs, d_in, totals_host, t_c, t_d, dev, stream)

    per_seg = []
    for i, t in enumerate(segs):
        per_seg.append({"segment": t.name, "elem_width": t.elem_width, "bytes": t.nbytes,
                        "ratio": round(t.nbytes / totals_host[i], 4),
                        "compress_gbs": round(t.nbytes / (t_c[i] * 1e-3) / 1e9, 1),
                        "decompress_gbs": round(t.nbytes / (t_d[i] * 1e-3) / 1e9, 1),
                        "compress_roofline_frac": round(alg[i] / (t_c[i] * 1e-3) / 1e9 / peak, 3),
                        "decompress_roofline_frac": round(alg[i] / (t_d[i] * 1e-3) / 1e9 / peak, 3)})

    cpu = None
    if rank == 0:
        nb, tcpu_c, tcpu_d = cpu_oracle_sample(segs, args.cpu_sample_mib)
        cpu = {"value": nb / (tcpu_c + tcpu_d) / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"first {args.cpu_sample_mib:g} MiB of each of the {nseg} segments of the workload, compress + "
                         f"decompress, single thread",
               "compress_gbs": nb / tcpu_c / 1e9, "decompress_gbs": nb / tcpu_d / 1e9}
        if args.cpu_parallel_mib > 0:
            nb, tcpu_c, tcpu_d, threads = cpu_oracle_parallel(segs, args.cpu_parallel_mib)
            cpu["parallel"] = {
                "value": nb / (tcpu_c + tcpu_d) / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
                "sample": f"first {args.cpu_parallel_mib:g} MiB of each of the {nseg} segments, cut at chunk "
                          f"boundaries into one slice per thread, compress + decompress",
                "compress_gbs": nb / tcpu_c / 1e9, "decompress_gbs": nb / tcpu_d / 1e9}

    ms_per_step = elapsed_ms / args.steps
    if flush_buf is not None:  # the step's own calls, without the flushes between them
        ms_per_step = max_over_ranks(dist, tc_ms + td_ms, dev)
    value = world * raw / (ms_per_step * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u32", "data": "synthetic",
        "config": {"workload": workload_label(args.workload), "bytes_per_step_per_gpu": raw, "parallelism": f"replicas x{world}",
                   "l2": ("L2 flushed (256 MiB write) before every timed call; value from the calls' CUDA events"
                          if flush_buf is not None else "inputs larger than L2 (128-256 MiB per call); no flush"),
                   "sha256": {t.name: __import__("lossless_bit_plane_gb300.workloads", fromlist=["x"]).sha256(t.data)[:16]
                              for t in segs}},
        "compress_gbs": world * raw / (tc_ms * 1e-3) / 1e9,
        "decompress_gbs": world * raw / (td_ms * 1e-3) / 1e9,
        "ratio": raw / comp,
        "roofline": {"bound": "hbm", "kernel": dominant, "achieved": ach, "peak": peak, "unit": "GB/s",
                     "frac": ach / peak, "peak_kind": peak_kind,
                     "traffic": (encoder_traffic() if dominant == "pz_encode" and args.workload == "sweep"
                                 else None),
                     "encode_frac": comp_ach / peak, "decode_frac": dec_ach / peak},
        "cpu_baseline": cpu,
        "e2e": e2e,
        # per step: one encoder launch per compress call; per decompress call
        # the chunk-size group sums (inputs over 2048 chunks), a walk and a decode
        "gpu_launches": args.steps * launches_per_step,
        "clocks": clk,
        "segments": per_seg,
        "eq2": eq2(raw / comp, raw / (tc_ms * 1e-3) / 1e9),
        "size_only": sizes["size_only"],
        "ablation": sizes["ablation"],
        "swap": swap,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def run_sizes(args, segs, d_in, totals_host, dev, stream):
    """Outside the headline's timed region: the sizes-only entry point
    (pz_compressed_size) timed over the same segments, every chunk and every
    fourth chunk (the paper's sampling of large tensors), and the codec
    ablation of the paper's Fig. 3 -- the exact ratio of each single-encoding
    candidate mask and of BF16 coded with 32-bit symbols, over the sweep's
    activation segments (the uniform-random segment is left out)."""
    import torch

    from lossless_bit_plane_gb300 import _lib

    sh = stream.cuda_stream
    n = len(segs)
    d_tot = torch.zeros(n, dtype=torch.int64, device=dev)

    def sizes_all(stride, mask=_lib.PZ_CAND_ALL, width=None):
        for i, t in enumerate(segs):
            rc = _lib.pz_compressed_size(d_in[i].data_ptr(), t.nbytes, width or t.elem_width, mask, stride, 0,
                                         d_tot[i:i + 1].data_ptr(), sh)
            assert rc == 0, rc

    def timed(stride, reps):
        for _ in range(2):
            sizes_all(stride)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(reps):
            sizes_all(stride)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    raw = sum(t.nbytes for t in segs)
    reps = max(1, min(args.steps, 5))
    ms1 = timed(1, reps)
    tot1 = d_tot.cpu().tolist()
    assert tot1 == totals_host, "sizes-only totals differ from the compressed streams"
    ms4 = timed(4, reps)
    tot4 = d_tot.cpu().tolist()
    sampled_raw = sum(min(t.nbytes - 4096 * c, 4096) for t in segs for c in range(0, (t.nbytes + 4095) // 4096, 4))
    size_only = {"unit": "GB/s", "gbs": raw / (ms1 * 1e-3) / 1e9, "sampled_every_4th_gbs": raw / (ms4 * 1e-3) / 1e9,
                 "ratio": raw / sum(tot1), "sampled_ratio_estimate": sampled_raw / sum(tot4),
                 "launches_per_pass": n}

    groups = {"fp32": [i for i, t in enumerate(segs) if t.elem_width == 4 and not t.name.startswith("random")],
              "bf16": [i for i, t in enumerate(segs) if t.elem_width == 2]}
    masks = {"planezip": _lib.PZ_CAND_ALL, "zvc": _lib.PZ_CAND_ZVC, "bpc_dbx": _lib.PZ_CAND_DBX,
             "bx": _lib.PZ_CAND_BX, "zbx": _lib.PZ_CAND_ZBX}
    ablation = {"source": "Section V-A, Fig. 3 (single encodings vs the per-block choice; BF16 with 32-bit "
                          "symbols); ratios over the sweep's activation segments, uniform-random excluded"}
    for g, idx in groups.items():
        if not idx:
            continue
        graw = sum(segs[i].nbytes for i in idx)
        row = {}
        for name, m in masks.items():
            sizes_all(1, m)
            tot = d_tot.cpu().tolist()
            row[name] = round(graw / sum(tot[i] for i in idx), 4)
        row["best_single"] = max(row[k] for k in ("zvc", "bpc_dbx", "bx", "zbx"))
        if g == "bf16":
            sizes_all(1, _lib.PZ_CAND_ALL, width=4)
            tot = d_tot.cpu().tolist()
            row["planezip_with_32bit_symbols"] = round(graw / sum(tot[i] for i in idx), 4)
        ablation[g] = row
    return {"size_only": size_only, "ablation": ablation}


def run_swap(segs, d_in, totals_host, t_c, t_d, dev, stream, piece=64 << 20, slot=4 << 20):
    """Outside the headline's timed region: the compressed swap path on a few
    segments (a first piece of 32 MiB, then pieces of 64 MiB;
    pinned host memory), into one host buffer (pz_swap_out / pz_swap_in) and
    into a pool of 4 MiB host slots (pz_pool_*), against the plain pinned copy
    of the same bytes over the host link, with the paper's Equation 2
    evaluated on the measured numbers: x_t = min(m/g, max(m/(c g), m/B)) with
    g the plain copy's rate, c the ratio and B the codec's rate on that
    segment (raw bytes / kernel time)."""
    import torch

    from lossless_bit_plane_gb300 import _lib

    pick = []
    for pref in ("relu_fp32", "attention_bf16", "random"):
        pick += [i for i, t in enumerate(segs) if t.name.startswith(pref)][:1]
    if not pick:
        return None
    nmax = max(segs[i].nbytes for i in pick)
    h_raw = torch.empty(nmax, dtype=torch.uint8).pin_memory()
    bufs = _lib.SwapBuffers(nmax, piece, dev)
    pool = _lib.SwapPool(_lib.pz_swap_capacity(nmax, piece) + 2 * slot + (1 << 20), slot, piece, dev)
    back = torch.empty(nmax, dtype=torch.uint8, device=dev)

    def wall(fn, reps=3):
        fn()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(reps):
            fn()
        torch.cuda.synchronize()
        return (time.perf_counter() - t0) / reps

    def pool_out(x, ew):
        t, _ = pool.swap_out(x, ew)
        pool.release(t)

    rows = []
    for i in pick:
        t, x = segs[i], d_in[i]
        n = t.nbytes
        g_out = n / wall(lambda: h_raw[:n].copy_(x, non_blocking=True)) / 1e9
        g_in = n / wall(lambda: back[:n].copy_(h_raw[:n], non_blocking=True)) / 1e9
        length = bufs.swap_out(x, t.elem_width)
        s_out = n / wall(lambda: bufs.swap_out(x, t.elem_width)) / 1e9
        s_in = n / wall(lambda: bufs.swap_in(length, back[:n])) / 1e9
        ok = int(bufs.status.item()) == 0 and torch.equal(back[:n], x)
        p_out = n / wall(lambda: pool_out(x, t.elem_width)) / 1e9
        tensor, stored = pool.swap_out(x, t.elem_width)
        p_in = n / wall(lambda: pool.swap_in(tensor, back[:n])) / 1e9
        ok = ok and int(pool.status.item()) == 0 and torch.equal(back[:n], x)
        pool.release(tensor)
        c = n / totals_host[i]
        b_c, b_d = n / (t_c[i] * 1e-3) / 1e9, n / (t_d[i] * 1e-3) / 1e9
        eq2 = lambda g, b: 1.0 / min(1.0 / g, max(1.0 / (c * g), 1.0 / b))  # noqa: E731  (GB/s of raw bytes)
        e_out, e_in = eq2(g_out, b_c), eq2(g_in, b_d)
        rows.append({"segment": t.name, "ratio": round(c, 4), "container_bytes": length, "pool_stored_bytes": stored,
                     "link_d2h_gbs": round(g_out, 1), "link_h2d_gbs": round(g_in, 1),
                     "swap_out_gbs": round(s_out, 1), "swap_in_gbs": round(s_in, 1),
                     "pool_swap_out_gbs": round(p_out, 1), "pool_swap_in_gbs": round(p_in, 1),
                     "eq2_out_gbs": round(e_out, 1), "eq2_in_gbs": round(e_in, 1),
                     "swap_out_of_eq2": round(s_out / e_out, 3), "swap_in_of_eq2": round(s_in / e_in, 3),
                     "swap_out_of_link": round(s_out / g_out, 3), "swap_in_of_link": round(s_in / g_in, 3),
                     "round_trip_exact": ok})
    return {"max_piece_bytes": piece, "pool_slot_bytes": slot, "unit": "GB/s of raw bytes",
            "host_memory": "pinned", "segments": rows}


def count_launches(step) -> int:
    """This library's kernel launches in one step, counted from a CUDA
    activity trace of one extra, untimed step (the kernel names carry the
    library's namespace)."""
    import torch
    from torch.profiler import ProfilerActivity, profile

    with profile(activities=[ProfilerActivity.CUDA]):  # the first trace of a process may miss kernels
        torch.ones(1, device="cuda").add_(1)
        torch.cuda.synchronize()
    with profile(activities=[ProfilerActivity.CUDA]) as prof:
        step()
        torch.cuda.synchronize()
    return sum(1 for e in prof.events()
               if e.device_type == torch.autograd.DeviceType.CUDA and e.name.startswith(("pz::", "void pz::")))


def run_e2e(args, segs, d_out, d_back, d_tot, d_st, totals_host, dev, stream, world, dist):
    """Same round trip through the C ABI, but every step copies each segment's
    input from pinned host memory to the device and reads the compressed
    sizes and decode statuses back to the host at the end. The copies run on
    a second stream, so segment i+1 crosses the host link while segment i is
    compressed and decompressed; a copy into an input buffer waits until the
    previous step's compress has read it."""
    import torch

    from lossless_bit_plane_gb300 import _lib

    h_in = [torch.from_numpy(t.data).pin_memory() for t in segs]
    d_in = [torch.empty(t.nbytes, dtype=torch.uint8, device=dev) for t in segs]
    h_res = torch.empty(2 * len(segs), dtype=torch.int64).pin_memory()
    sh = stream.cuda_stream
    copy = torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in segs]    # input i is on the device
    ev_read = [torch.cuda.Event() for _ in segs]  # the compress of input i is done
    start = torch.cuda.Event()

    def step(first):
        start.record(stream)
        copy.wait_event(start)
        for i, t in enumerate(segs):
            with torch.cuda.stream(copy):
                if not first:
                    copy.wait_event(ev_read[i])
                d_in[i].copy_(h_in[i], non_blocking=True)
                ev_in[i].record(copy)
        for i, t in enumerate(segs):
            stream.wait_event(ev_in[i])
            rc = _lib.pz_compress(d_in[i].data_ptr(), t.nbytes, t.elem_width, d_out[i].data_ptr(), d_out[i].numel(),
                                  d_tot[i:i + 1].data_ptr(), sh)
            assert rc == 0
            ev_read[i].record(stream)
            rc = _lib.pz_decompress(d_out[i].data_ptr(), int(totals_host[i]), t.elem_width, d_back[i].data_ptr(),
                                    t.nbytes, d_st[i:i + 1].data_ptr(), sh)
            assert rc == 0
        h_res[: len(segs)].copy_(d_tot, non_blocking=True)
        h_res[len(segs):].copy_(d_st.to(torch.int64), non_blocking=True)

    for w in range(max(1, args.warmup)):
        step(w == 0)
    torch.cuda.synchronize()
    barrier(dist)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        step(False)
    t1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(dist, t0.elapsed_time(t1) / args.steps, dev)
    assert h_res[: len(segs)].tolist() == totals_host and h_res[len(segs):].tolist() == [0] * len(segs)
    for i in range(len(segs)):
        assert torch.equal(d_back[i], d_in[i]), f"end-to-end round trip failed on segment {i}"
    raw = sum(t.nbytes for t in segs)
    return {"value": world * raw / (ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": ms,
            "h2d_bytes_per_step": raw, "d2h_bytes_per_step": 16 * len(segs),
            "overlap": "host-to-device copies on a second stream, overlapped with the codec"}


def eq2(ratio: float, bce_gbs: float, gammas=(24.0, 450.0)):
    """The paper's effective transfer time x_t = min(m/g, max(m/(c g), m/B_CE))
    (Section III-C, Eq. 2) per GiB, for the measured ratio c and compress rate
    B_CE, at the paper's PCIe 4.0 24 GB/s and at an assumed 450 GB/s per
    direction for GB300's NVLink-C2C host link."""
    m = float(1 << 30)
    out = {}
    for g in gammas:
        x = min(m / (g * 1e9), max(m / (ratio * g * 1e9), m / (bce_gbs * 1e9)))
        out[f"gamma_{g:g}GBps"] = {"x_t_ms_per_GiB": 1e3 * x, "uncompressed_ms_per_GiB": 1e3 * m / (g * 1e9)}
    return out


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, rank)
    return run_ours(args, rank, world, local)


if __name__ == "__main__":
    sys.exit(main())
