#!/usr/bin/env python
"""Benchmark of the paged GQA decode step on GB300.

One step = one pass of the hot path over one batch: kv_append of the newest
token of every sequence, then paged decode attention over every cached
position (context includes the appended token), issued as one C-ABI call
(pgd_append_decode_attention).  Default workload:
batch 16, context 8192, 32 query / 8 KV heads, d 128, block 16, bf16
(512 MiB of K/V per step, larger than the 129 MB L2, so no flush is needed).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--splits S] [--impl ours|reference]

Prints one JSON line (rank 0).  value = algorithmic K/V bytes read per step
summed over ranks / max-over-ranks time, in GB/s (1e9 B/s).  Under torchrun
(N > 1) every rank runs an independent replica of the workload on its own GPU
(the path shards by sequence and KV head with no exchange); timing
collectives use gloo on the host.  --impl reference times the float64 CPU
oracle on a bounded sample of the same workload, on rank 0 only.
"""
from __future__ import annotations

import argparse
import hashlib
import json
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

METRIC = "paged decode attention KV GB/s and % of GB300 HBM peak; seq-layer-steps/sec"
NOMINAL_HBM_GBS = 8000.0     # nominal GB300 HBM3e bandwidth (~8 TB/s)
FALLBACK_HBM_GBS = 6800.0    # profiling recipe's fallback when no measured peak exists
L2_BYTES = 129 * 10**6
ATTENTION_SOURCES = [os.path.join(ROOT, "paged_gqa_decode_kv_gb300", "csrc", f)
                     for f in ("attention_kernel.cuh", "pgd_device.cuh")]
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "paged_attention_batch16_ctx8192.md")
PROFILE_SUMMARY_FP8 = os.path.join(ROOT, "profiles", "paged_attention_fp8_batch16_ctx8192.md")
MLA_SOURCES = [os.path.join(ROOT, "paged_gqa_decode_kv_gb300", "csrc", f)
               for f in ("mla_attention.cu", "attention_kernel.cuh", "pgd_device.cuh")]
PROFILE_SUMMARY_MLA = os.path.join(ROOT, "profiles", "mla_attention_batch16_ctx8192_h128.md")
SHORT_SOURCES = [os.path.join(ROOT, "paged_gqa_decode_kv_gb300", "csrc", f)
                 for f in ("short_attention.cu", "short_attention.cuh", "kv_quant.cuh",
                           "pgd_device.cuh")]
PROFILE_SUMMARY_SHORT = os.path.join(ROOT, "profiles", "short_attention_single_ctx512.md")


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--workload", default="batch16_ctx8192")
    ap.add_argument("--splits", type=int, default=0, help="0 = automatic")
    ap.add_argument("--cascade", action="store_true",
                    help="shared-prefix workloads: read each shared prefix once per group "
                         "(pgd_cascade_decode_attention)")
    ap.add_argument("--verify", type=int, default=0, metavar="T",
                    help="speculative verify: T new query tokens per sequence (appended with "
                         "pgd_kv_append_tokens, attended causally with pgd_paged_verify_attention)")
    ap.add_argument("--mla", action="store_true",
                    help="MLA latent-cache decode (workloads mla128_batch16_ctx8192, "
                         "mla128_batch64_ctx4096; default the first)")
    ap.add_argument("--kv", choices=["bf16", "fp8"], default="bf16",
                    help="cache format: bf16, or FP8 E4M3 codes + per-(token, head) scales")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    return ap.parse_args(argv)


# ------------------------------------------------------------ distribution
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def dist_init(world: int):
    if world <= 1:
        return None
    import torch.distributed as dist
    if not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("gloo")
    return dist


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int) -> float:
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampling (every 100 ms) in the background."""
    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_id: str):
        self.samples = []
        self.proc = None
        self.thread = None
        self.gpu_id = gpu_id

    def start(self):
        cmd = ["nvidia-smi", "-i", self.gpu_id, "--query-gpu=" + ",".join(self.FIELDS),
               "--format=csv,noheader,nounits", "-lms", "100"]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                sm, smax = float(parts[0]), float(parts[1])
            except ValueError:
                continue
            active = [r for r, v in zip(self.REASONS, parts[3:]) if v.lower() == "active"]
            self.samples.append((time.time(), sm, smax, active))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        win = [s for s in self.samples if t0 <= s[0] <= t1]
        window = "warmup+timed"
        if not win:
            win = [s for s in self.samples if t0 <= s[0] <= t1 + 0.5]
            window = "warmup+timed+0.5s"
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "window": "none"}
        reasons = sorted({r for s in win for r in s[3]})
        return {"sm_mhz": statistics.median(s[1] for s in win),
                "sm_max_mhz": max(s[2] for s in win), "reasons": reasons,
                "samples": len(win), "window": window}


class NvmlClocks:
    """SM clock and clock-event reasons read in-process through NVML (read-only
    queries over ctypes) about every half millisecond in a background thread,
    so that a timed region of a few milliseconds still holds samples.
    Unavailable NVML leaves it empty (the nvidia-smi sampler stays)."""
    BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
            0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, gpu_uuid: str):
        import ctypes
        self.samples = []
        self.ok = False
        self._stop = threading.Event()
        self.thread = None
        try:
            L = ctypes.CDLL("libnvidia-ml.so.1")
            if L.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            if L.nvmlDeviceGetHandleByUUID(gpu_uuid.encode(), ctypes.byref(h)) != 0:
                return
            mx = ctypes.c_uint(0)
            L.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))
            self.max_mhz = float(mx.value)
            self.reasons_fn = getattr(L, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                L.nvmlDeviceGetCurrentClocksThrottleReasons
            self.L, self.h, self.ctypes = L, h, ctypes
            self.ok = True
        except (OSError, AttributeError):
            self.ok = False

    def _run(self):
        c, L, h = self.ctypes, self.L, self.h
        mhz, bits = c.c_uint(0), c.c_ulonglong(0)
        while not self._stop.is_set():
            if L.nvmlDeviceGetClockInfo(h, 1, c.byref(mhz)) == 0 and \
                    self.reasons_fn(h, c.byref(bits)) == 0:
                self.samples.append((time.time(), float(mhz.value), int(bits.value)))
            time.sleep(0.0005)

    def start(self):
        if self.ok:
            self.thread = threading.Thread(target=self._run, daemon=True)
            self.thread.start()

    def stop(self):
        self._stop.set()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        win = [s for s in self.samples if t0 <= s[0] <= t1]
        if not win:
            return None
        reasons = sorted({n for s in win for b, n in self.BITS.items() if s[2] & b})
        return {"sm_mhz": statistics.median(s[1] for s in win), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(win), "window": "timed steps",
                "source": "NVML in-process, ~0.5 ms period"}


def clocks_record(smi, nvml, t_wall0, t_wall1, t_timed0, t_timed1):
    """The clock record of a run: NVML samples inside the timed steps when
    there are any, else the nvidia-smi samples; both kept."""
    smi_sum = smi.summary(t_wall0, t_wall1)
    nv = nvml.summary(t_timed0, t_timed1) if nvml is not None else None
    if nv is None:
        return smi_sum
    return dict(nv, nvidia_smi=smi_sum)


# ------------------------------------------------------------------- peaks
def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def profiled_traffic(kv: str = "bf16", workload: str = "batch16_ctx8192", short: bool = False):
    """DRAM bytes per launch from the committed ncu summary of the attention
    kernel on this workload, or None if there is none or the kernel source
    changed since that capture."""
    if short:
        if workload != "single_ctx512" or kv != "bf16":
            return None
        path, sources = PROFILE_SUMMARY_SHORT, SHORT_SOURCES
    elif workload == "batch16_ctx8192":
        path, sources = (PROFILE_SUMMARY_FP8 if kv == "fp8" else PROFILE_SUMMARY), None
    else:
        return None
    try:
        text = open(path).read()
    except OSError:
        return None
    m_bytes = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
    m_sha = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    if not (m_bytes and m_sha):
        return None
    return int(m_bytes.group(1)) if kernel_source_sha256(sources) == m_sha.group(1) else None


def kernel_source_sha256(paths=None) -> str:
    """sha256 of a kernel's sources (default: the attention kernel's,
    attention_kernel.cuh, then the device header it includes)."""
    h = hashlib.sha256()
    for path in (paths or ATTENTION_SOURCES):
        h.update(open(path, "rb").read())
    return h.hexdigest()


def profiled_mla_traffic(workload: str):
    """DRAM bytes per launch of the MLA attention kernel from its committed ncu
    summary (batch 16 x 8192 tokens), or None if the kernel changed since."""
    if workload != "mla128_batch16_ctx8192":
        return None
    try:
        text = open(PROFILE_SUMMARY_MLA).read()
    except OSError:
        return None
    m_bytes = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
    m_sha = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    if not (m_bytes and m_sha):
        return None
    return int(m_bytes.group(1)) if kernel_source_sha256(MLA_SOURCES) == m_sha.group(1) else None


# ------------------------------------------------------------ CPU baseline
def oracle_sample(pb_host, n_seq: int, n_threads: int = 0):
    """Run the oracle on the first n_seq sequences; return (seconds, bytes)."""
    import oracle
    from paged_gqa_decode_kv_gb300 import inputs
    q = pb_host["q"][:n_seq]
    t = pb_host["tables"][:n_seq]
    c = pb_host["lens"][:n_seq]
    t0 = time.perf_counter()
    if pb_host.get("T", 0):
        oracle.paged_verify_attention(q, pb_host["k"], pb_host["v"], t, c, pb_host["scale"],
                                      n_threads=n_threads)
        per_token = 2 * pb_host["n_kv"] * pb_host["d"] * 2
    elif pb_host["kv"] == "fp8":
        oracle.paged_attention_fp8(q, pb_host["k"], pb_host["v"], t, c, pb_host["scale"],
                                   pb_host["bs"], n_threads=n_threads)
        per_token = 2 * pb_host["n_kv"] * (pb_host["d"] + 4)
    else:
        oracle.paged_attention(q, pb_host["k"], pb_host["v"], t, c, pb_host["scale"],
                               n_threads=n_threads)
        per_token = 2 * pb_host["n_kv"] * pb_host["d"] * 2
    dt = time.perf_counter() - t0
    return dt, int(c.sum()) * per_token


def host_copy(pb, T: int = 0):
    """Host copies of a batch for the oracle.  Verify batches (T > 0) get the
    oracle's own append of their new tokens first (untimed)."""
    k, v = pb.k_cache.cpu(), pb.v_cache.cpu()
    if T:
        import oracle
        k, v = oracle.kv_append_tokens(k, v, pb.k_new.cpu(), pb.v_new.cpu(),
                                       pb.block_tables.cpu(), pb.positions.cpu())
    return {"q": pb.q.cpu(), "k": k, "v": v,
            "tables": pb.block_tables.cpu(), "lens": pb.context_lens.cpu(), "scale": pb.scale,
            "n_kv": pb.n_kv, "d": pb.head_dim, "B": pb.batch, "n_q": pb.q.shape[-2],
            "kv": pb.kv_format, "bs": pb.block_size, "T": T}


def cpu_baseline(pb_host, seconds: float):
    import oracle
    B = pb_host["B"]
    rows = B * pb_host["n_q"] * max(1, pb_host.get("T", 0))
    cores = oracle.threads_used(0, rows)
    total_t, total_b, calls = 0.0, 0, 0
    while total_t < seconds and calls < 200:
        dt, nb = oracle_sample(pb_host, B)
        total_t += dt
        total_b += nb
        calls += 1
    one = one_thread_baseline(pb_host, min(5.0, seconds / 2))
    return {"value": round(total_b / total_t / 1e9, 4), "unit": "GB/s", "cores": cores,
            "kind": "oracle", "one_thread": one,
            "sample": "float64 oracle %s over the full batch (all %d sequences, %d query "
                      "heads), %d call(s), %.1f s; kv_append excluded (a %d-byte copy)"
                      % ("verify attention (%d query tokens per sequence)" % pb_host["T"]
                         if pb_host.get("T", 0) else "attention", B, pb_host["n_q"], calls,
                         total_t, 2 * B * max(1, pb_host.get("T", 0)) * pb_host["n_kv"] * 256)}


def one_thread_baseline(pb_host, seconds: float):
    """The oracle on one host thread over the first sequence, repeated for
    about `seconds`."""
    total_t, total_b, calls = 0.0, 0, 0
    while total_t < seconds and calls < 100:
        dt, nb = oracle_sample(pb_host, 1, n_threads=1)
        total_t += dt
        total_b += nb
        calls += 1
    return {"value": round(total_b / total_t / 1e9, 4), "unit": "GB/s", "cores": 1,
            "sample": "float64 oracle over the first sequence (all %d query heads), one "
                      "thread, %d call(s), %.1f s" % (pb_host["n_q"], calls, total_t)}


# ------------------------------------------------- read-only streaming peak
READ_ONLY_BYTES = 2 << 30     # 2 GiB, > 15 x L2


def read_only_peak(dev, stream, passes: int = 10):
    """GB/s of the library's read-only streaming pass (pgd_read_stream) over a
    2 GiB buffer, both access patterns (16-byte loads; 4 KiB bulk copies into
    shared memory, the attention kernels' pattern), each the best and the mean
    of `passes` CUDA-event-timed passes.  Returns (best of both, record)."""
    import torch
    import paged_gqa_decode_kv_gb300 as pgd
    buf = torch.ones(READ_ONLY_BYTES // 4, dtype=torch.int32, device=dev)
    rec = {}
    for mode, name in ((0, "loads16"), (1, "bulk4k")):
        for _ in range(3):
            pgd.read_stream(buf, mode, stream=stream)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(passes)]
        for a, b in evs:
            a.record(stream)
            pgd.read_stream(buf, mode, stream=stream)
            b.record(stream)
        torch.cuda.synchronize()
        ms = [a.elapsed_time(b) for a, b in evs]
        rec[name] = {"gbs_best": round(READ_ONLY_BYTES / (min(ms) / 1e3) / 1e9, 1),
                     "gbs_mean": round(READ_ONLY_BYTES / (statistics.fmean(ms) / 1e3) / 1e9, 1)}
    flags = pgd.device_errors(clear=True, stream=stream)
    if flags:
        raise RuntimeError("device error word %d after the read-only passes" % flags)
    del buf
    best = max(r["gbs_best"] for r in rec.values())
    rec.update({"bytes": READ_ONLY_BYTES, "passes": passes, "kernel": "pgd_read_stream"})
    return best, rec


# ------------------------------------------------------ CUDA-graph replay
def graph_steps(step_on, K: int, bytes_per_step: int, world: int):
    """The same steps (the same C-ABI calls) captured into one CUDA graph of
    up to 64 steps and replayed: the device-side step time without the host's
    per-call launch cost.  A side figure, not the headline.  None if the
    capture fails (its error is then reported)."""
    import torch
    n = max(1, min(K, 64))
    reps = max(1, -(-K // n))
    try:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(3):
                step_on(side)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            cs = torch.cuda.current_stream()
            for _ in range(n):
                step_on(cs)
        g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        a.record()
        for _ in range(reps):
            g.replay()
        b.record()
        torch.cuda.synchronize()
        barrier(world)
        ms = max_over_ranks(a.elapsed_time(b), world) / (reps * n)
        del g
        return {"ms_per_step": round(ms, 5),
                "value": round(sum_over_ranks(bytes_per_step, world) / (ms / 1e3) / 1e9, 2),
                "unit": "GB/s", "steps": reps * n,
                "note": "%d steps per graph, %d replays; side figure" % (n, reps)}
    except Exception as exc:  # capture unsupported: report, do not fail the run
        return {"error": str(exc)[:200]}


# ------------------------------------------ PyTorch gather + SDPA (context)
def torch_sdpa_context(pb, kv_bytes: int, iters: int, stream, ours):
    """Context only (not the oracle, not a target): the same attention in
    plain PyTorch on the GPU -- gather every sequence's blocks through the
    block table from a row-major copy of the pool, then
    scaled_dot_product_attention with GQA and a length mask."""
    import torch
    import torch.nn.functional as F
    from paged_gqa_decode_kv_gb300 import inputs
    B, n_q, d = pb.q.shape
    n_kv, bs = pb.n_kv, pb.block_size
    MB = pb.block_tables.shape[1]
    L = MB * bs
    # untimed preparation: row-major pools with the never-read slots zeroed
    # (NaN there would reach the masked product)
    kr = torch.nan_to_num(inputs.untile_pool(pb.k_cache).contiguous(), nan=0.0)
    vr = torch.nan_to_num(inputs.untile_pool(pb.v_cache).contiguous(), nan=0.0)
    tab = pb.block_tables.clamp(min=0).long()
    lens = pb.context_lens.long()
    mask = None
    if int(lens.min()) != L:
        mask = (torch.arange(L, device=tab.device)[None, :] < lens[:, None]).view(B, 1, 1, L)
    q4 = pb.q.view(B, n_q, 1, d)

    def run():
        k = kr[tab].permute(0, 2, 1, 3, 4).reshape(B, n_kv, L, d)
        v = vr[tab].permute(0, 2, 1, 3, 4).reshape(B, n_kv, L, d)
        return F.scaled_dot_product_attention(q4, k, v, attn_mask=mask, scale=pb.scale,
                                              enable_gqa=True)

    with torch.cuda.stream(stream):
        for _ in range(3):
            o = run()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(iters):
            o = run()
        b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / iters
    diff = (o.view(B, n_q, d).float() - ours.float()).abs().max().item()
    del kr, vr
    return {"kind": "context: PyTorch on the GPU (block gather by advanced indexing from a "
                    "row-major copy of the pool, then scaled_dot_product_attention with "
                    "enable_gqa and a length mask); not the oracle, not a target",
            "ms_per_step": round(ms, 5), "gbs": round(kv_bytes / (ms / 1e3) / 1e9, 2),
            "iters": iters, "max_abs_diff_vs_ours": round(diff, 5)}


# --------------------------------------------------------------- our arm
def config_block(pb, name, splits, n_pools):
    return {"workload": name, "batch": pb.batch, "context": sorted(set(pb.context_lens.tolist()))
            if pb.batch <= 4 else "%d..%d" % (int(pb.context_lens.min()),
                                              int(pb.context_lens.max())),
            "n_q": pb.n_q, "n_kv": pb.n_kv, "head_dim": pb.head_dim,
            "block_size": pb.block_size,
            "kv_dtype": "bf16" if pb.kv_format == "bf16" else
            "fp8_e4m3 codes + fp32 scale per (token, head)",
            "splits": "auto" if splits == 0 else splits,
            "kv_layout": "tiled 8x8 core matrices per (block, head)" if pb.kv_format == "bf16"
            else "per 8-token group: 8x16-byte core matrices of codes, then 8 scales",
            "l2": ("K/V pool %.0f MB > 129 MB L2, no flush" % (pool_bytes(pb) / 1e6))
            if n_pools == 1 else
            ("%d copies of the %.1f MB K/V pool rotated step by step (%.0f MB > 2 x L2), "
             "no flush" % (n_pools, pool_bytes(pb) / 1e6, n_pools * pool_bytes(pb) / 1e6))}


def pool_bytes(pb) -> int:
    return 2 * pb.k_cache.numel() * pb.k_cache.element_size()


def pool_copies(pb) -> int:
    """Copies of the K/V pool to rotate through so that no step finds the
    previous step's blocks in L2: one when the pool alone exceeds twice the
    L2, else enough copies to exceed it."""
    b = pool_bytes(pb)
    return 1 if b > 2 * L2_BYTES else -(-2 * L2_BYTES // b)


def run_ours(args, rank, world, local):
    import torch

    import __graft_entry__
    import paged_gqa_decode_kv_gb300 as pgd
    from paged_gqa_decode_kv_gb300 import inputs

    __graft_entry__.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    T = args.verify
    if T:
        if args.kv != "bf16" or args.cascade:
            raise SystemExit("--verify needs the bf16 cache and no --cascade")
        vb = inputs.make_verify_workload(args.workload, T, device=dev)
        pb = vb.paged
        pb.q, pb.k_new, pb.v_new, pb.positions = vb.q, vb.k_new, vb.v_new, vb.positions
    else:
        pb = inputs.make_workload(args.workload, device=dev, append=True, kv_format=args.kv)
    B, n_q, n_kv = pb.batch, pb.q.shape[-2], pb.n_kv
    fp8 = args.kv == "fp8"
    append_attend = pgd.append_decode_attention_fp8 if fp8 else pgd.append_decode_attention
    attend = pgd.paged_decode_attention_fp8 if fp8 else pgd.paged_decode_attention
    if args.cascade:
        if fp8 or not pb.shared_blocks:
            raise SystemExit("--cascade needs a bf16 shared-prefix workload")
        groups = inputs.prefix_groups(pb, [(0, B, pb.shared_blocks)])
        cws = torch.zeros(pgd.cascade_workspace_size(B, n_q, n_kv, pb.block_size, groups[4],
                                                     groups[5], args.splits),
                          dtype=torch.uint8, device=dev)

        def attend(out_, q_, kc, vc, tables, lens, scale, num_splits=0, workspace=None,
                   stream=None):
            return pgd.cascade_decode_attention(out_, q_, kc, vc, tables, lens, *groups[:4],
                                                groups[4], groups[5], scale,
                                                num_splits=num_splits, workspace=cws,
                                                stream=stream)

        def append_attend(out_, q_, kn, vn, kc, vc, tables, lens, scale, num_splits=0,
                          workspace=None, stream=None):
            pgd.kv_append(kn, vn, kc, vc, tables, pb.positions, stream=stream)
            return attend(out_, q_, kc, vc, tables, lens, scale, num_splits=num_splits,
                          stream=stream)
    if T:
        ws = torch.zeros(max(1, pgd.verify_workspace_size(B, T, n_q, n_kv, args.splits)),
                         dtype=torch.uint8, device=dev)

        def attend(out_, q_, kc, vc, tables, lens, scale, num_splits=0, workspace=None,
                   stream=None):
            return pgd.paged_verify_attention(out_, q_, kc, vc, tables, lens, scale,
                                              num_splits=num_splits, workspace=ws, stream=stream)

        def append_attend(out_, q_, kn, vn, kc, vc, tables, lens, scale, num_splits=0,
                          workspace=None, stream=None):
            pgd.kv_append_tokens(kn, vn, kc, vc, tables, pb.positions, stream=stream)
            return attend(out_, q_, kc, vc, tables, lens, scale, num_splits=num_splits,
                          stream=stream)
    else:
        ws = pgd.make_workspace(B, n_q, n_kv, args.splits, dev)
    out = torch.empty_like(pb.q)
    # Short contexts (every context within 1024 tokens, at most 128 units)
    # run the short-context kernel: one launch, the append fused.
    short = (not args.cascade and not T and
             pgd.uses_short_path(B, n_kv, pb.block_size, pb.block_tables.shape[1], args.splits))
    grid = (8 * B * n_kv) if short else pgd.attention_grid(B, n_q, n_kv, pb.block_size,
                                                            args.splits)
    stream = torch.cuda.current_stream()
    # Headline bytes: each physical block once (equal to the logical bytes
    # unless sequences share prefix blocks, whose re-reads may hit L2).
    kv_bytes = inputs.kv_bytes_read(pb, unique=True)
    kv_bytes_logical = inputs.kv_bytes_read(pb)
    n_pools = pool_copies(pb)
    pools = [(pb.k_cache, pb.v_cache)] + [(pb.k_cache.clone(), pb.v_cache.clone())
                                          for _ in range(n_pools - 1)]
    it = [0]

    def next_pool():
        kc, vc = pools[it[0] % n_pools]
        it[0] += 1
        return kc, vc

    # The plain decode paths time prepared C-ABI calls (arguments checked and
    # marshalled once per pool copy): the Python side of a regular binding
    # call costs about 10 us, more than a short-context step on the GPU.
    # (multi-query verify: the one-call append + verify step, whose attention
    # alone goes through the binding)
    prepared = not args.cascade
    prepared_attn = prepared and not T
    if prepared:
        op = "_fp8" if fp8 else ""
        step_op = "append_verify_attention" if T else "append_decode_attention" + op
        step_calls = [pgd.prepare(step_op, out, pb.q, pb.k_new, pb.v_new,
                                  kc, vc, pb.block_tables, pb.context_lens, pb.scale,
                                  num_splits=args.splits, workspace=ws, stream=stream)
                      for kc, vc in pools]
    if prepared_attn:
        attn_calls = [pgd.prepare("paged_decode_attention" + op, out, pb.q, kc, vc,
                                  pb.block_tables, pb.context_lens, pb.scale,
                                  num_splits=args.splits, workspace=ws, stream=stream)
                      for kc, vc in pools]

    def step():
        # kv_append at context_lens - 1, then attention: one C-ABI call
        if prepared:
            step_calls[it[0] % n_pools]()
            it[0] += 1
            return
        kc, vc = next_pool()
        append_attend(out, pb.q, pb.k_new, pb.v_new, kc, vc, pb.block_tables, pb.context_lens,
                      pb.scale, num_splits=args.splits, workspace=ws, stream=stream)

    def attention_only():
        if prepared_attn:
            attn_calls[it[0] % n_pools]()
            it[0] += 1
            return
        kc, vc = next_pool()
        attend(out, pb.q, kc, vc, pb.block_tables, pb.context_lens, pb.scale,
               num_splits=args.splits, workspace=ws, stream=stream)

    gpu_uuid = "GPU-" + str(torch.cuda.get_device_properties(local).uuid)
    sampler = ClockSampler(gpu_uuid)
    sampler.start()
    nvml = NvmlClocks(gpu_uuid)
    nvml.start()
    time.sleep(0.3)
    t_wall0 = time.time()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    flags = pgd.device_errors(clear=True, stream=stream)
    if flags:
        raise RuntimeError("device error word %d after warm-up" % flags)

    K = args.steps
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t_timed0 = time.time()
    e0.record(stream)
    for i in range(K):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    t_timed1 = time.time()
    barrier(world)
    # The attention kernel alone, K launches each between two events on its
    # stream (inputs > L2, so every launch streams from HBM): the duration
    # behind the roofline figure.
    ev_a = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev_b = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for i in range(K):
        ev_a[i].record(stream)
        attention_only()
        ev_b[i].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    t_wall1 = time.time()
    time.sleep(0.25)
    sampler.stop()
    nvml.stop()
    elapsed_ms = e0.elapsed_time(e1)
    attn_all = [a.elapsed_time(b) for a, b in zip(ev_a, ev_b)]
    attn_ms = statistics.fmean(attn_all)
    attn_med = statistics.median(attn_all)
    flags = pgd.device_errors(clear=True, stream=stream)
    if flags:
        raise RuntimeError("device error word %d after the timed steps" % flags)

    max_ms = max_over_ranks(elapsed_ms, world)
    total_bytes = sum_over_ranks(kv_bytes * K, world)
    value = total_bytes / (max_ms / 1e3) / 1e9
    seq_steps = sum_over_ranks(B * K, world) / (max_ms / 1e3)

    # end to end through the C ABI with host (pinned) inputs and outputs
    q_h = pb.q.cpu().pin_memory()
    kn_h, vn_h = pb.k_new.cpu().pin_memory(), pb.v_new.cpu().pin_memory()
    cl_h = pb.context_lens.cpu().pin_memory()
    out_h = torch.empty_like(q_h).pin_memory()
    q_d, kn_d, vn_d = torch.empty_like(pb.q), torch.empty_like(pb.k_new), torch.empty_like(pb.v_new)
    cl_d = torch.empty_like(pb.context_lens)
    out_d = torch.empty_like(pb.q)

    if prepared:
        e2e_calls = [pgd.prepare("verify_step" if T else "decode_step", out_h, q_h, kn_h, vn_h,
                                 cl_h, out_d, q_d, kn_d, vn_d, cl_d, kc, vc, pb.block_tables,
                                 pb.scale, args.splits, ws, stream=stream) for kc, vc in pools]

    def e2e_step():
        if prepared:
            e2e_calls[it[0] % n_pools]()
            it[0] += 1
            return
        kc, vc = next_pool()
        pgd.decode_step(out_h, q_h, kn_h, vn_h, cl_h, out_d, q_d, kn_d, vn_d, cl_d, kc, vc,
                        pb.block_tables, pb.scale, args.splits, ws, stream=stream)

    for _ in range(args.warmup):
        e2e_step()
    barrier(world)
    torch.cuda.synchronize()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(K):
        e2e_step()
    f1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = max_over_ranks(f0.elapsed_time(f1), world)
    e2e_value = total_bytes / (e2e_ms / 1e3) / 1e9
    h2d = (q_h.numel() + kn_h.numel() + vn_h.numel()) * 2 + cl_h.numel() * 4
    d2h = out_h.numel() * 2

    # Small working sets: the rotated pool copies above give the cold figure;
    # the same step on one copy every time (pool resident in L2) is the hot one.
    hot = None
    if n_pools > 1:
        kc0, vc0 = pools[0]

        def hot_step():
            if prepared:
                step_calls[0]()
                return
            append_attend(out, pb.q, pb.k_new, pb.v_new, kc0, vc0, pb.block_tables,
                          pb.context_lens, pb.scale, num_splits=args.splits, workspace=ws,
                          stream=stream)
        for _ in range(max(3, args.warmup)):
            hot_step()
        h0, h1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        h0.record(stream)
        for _ in range(K):
            hot_step()
        h1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        hot_ms = max_over_ranks(h0.elapsed_time(h1), world)
        hot = {"ms_per_step": round(hot_ms / K, 5),
               "value": round(total_bytes / (hot_ms / 1e3) / 1e9, 2), "unit": "GB/s",
               "note": "one %.1f MB pool copy every step (L2-resident after the first)"
                       % (pool_bytes(pb) / 1e6)}

    graph_rec = graph_steps(lambda st: append_attend(
        out, pb.q, pb.k_new, pb.v_new, *next_pool(), pb.block_tables, pb.context_lens, pb.scale,
        num_splits=args.splits, workspace=ws, stream=st), K, kv_bytes, world)
    ro_best, ro_rec = read_only_peak(dev, stream)
    ctx_rec = None
    if not fp8 and not T:
        ctx_rec = torch_sdpa_context(pb, kv_bytes, min(K, 50), stream, out)

    peak, peak_kind = hbm_peak()
    achieved = kv_bytes / (attn_ms / 1e3) / 1e9
    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(max_ms / K, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8_e4m3 (q.k^T), bf16 (p.v)" if fp8 else "bf16",
        "accumulate": "f32",
        "data": ("synthetic (seeded E4M3 K/V codes + per-token scales, N(0,1) bf16 Q, random "
                 "block tables)") if fp8 else
                "synthetic (seeded N(0,1) bf16 K/V/Q, random block tables)",
        "config": dict(config_block(pb, args.workload, args.splits, n_pools),
                       **({"cascade": True} if args.cascade else {}),
                       **({"verify_tokens": T} if T else {})),
        "grid_ctas": grid,
        "kv_bytes_per_step": kv_bytes,
        "kv_bytes_per_step_logical": kv_bytes_logical,
        "effective_logical_gbs": round(sum_over_ranks(kv_bytes_logical * K, world)
                                       / (max_ms / 1e3) / 1e9, 2),
        "seq_layer_steps_per_s": round(seq_steps, 1),
        "pct_of_hbm_peak": {"nominal_8tbs": round(100 * value / world / NOMINAL_HBM_GBS, 2),
                            peak_kind: round(100 * value / world / peak, 2),
                            "read_only": round(100 * value / world / ro_best, 2)},
        "read_only_stream": dict(ro_rec, gbs=ro_best),
        "roofline": {"bound": "hbm",
                     "kernel": ("pgd::pf::prefix_attention_kernel + pgd::tc::paged_attention_kernel"
                                " + pgd::pf::cascade_combine_kernel (cascade, tcgen05)")
                               if args.cascade else
                               ("pgd::tc::paged_attention_kernel<%d rows, bs, bf16> (tcgen05, "
                                "multi-query verify)" % (T * (n_q // n_kv))) if T else
                               ("pgd::sc::short_attention_kernel<G, bs, %s> (short contexts: "
                                "CUDA cores, cluster log-sum-exp merge; latency-bound)"
                                % ("fp8" if fp8 else "bf16")) if short else
                               "pgd::tc::paged_attention_kernel<G, bs, %s> (tcgen05)"
                               % ("fp8" if fp8 else "bf16"),
                     "achieved": round(achieved, 2), "peak": peak, "peak_kind": peak_kind,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": None if (args.cascade or T) else
                     profiled_traffic(args.kv, args.workload, short),
                     "launch_ms": round(attn_ms, 5), "launch_ms_median": round(attn_med, 5),
                     "bytes_per_launch": kv_bytes,
                     "frac_of_read_only": round(achieved / ro_best, 4)},
        "e2e": dict({"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                     "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms / K, 5)},
                    **({"path": "pgd_decode_step (host buffers; no cascade)"}
                       if args.cascade else
                       {"path": "pgd_verify_step (host buffers)"} if T else {})),
        # kv_append + attention (cascade: + the prefix pass and the combine;
        # the short-context kernel appends in the same launch)
        "gpu_launches": (4 if args.cascade else 1 if short else 2) * K,
        "host_call": ("prepared C-ABI call (pgd.prepare: arguments checked and marshalled once "
                      "per pool copy)") if prepared else "Python binding call per step",
        "clocks": clocks_record(sampler, nvml, t_wall0, t_wall1, t_timed0, t_timed1),
        "gpu": torch.cuda.get_device_name(local),
    }
    if hot is not None:
        result["cold"] = {"ms_per_step": result["ms_per_step"], "value": result["value"],
                          "unit": "GB/s", "note": "the headline: %d pool copies rotated"
                                                  % n_pools}
        result["hot"] = hot
    if ctx_rec is not None:
        result["torch_gather_sdpa"] = ctx_rec
    if graph_rec is not None:
        result["graph"] = graph_rec
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(host_copy(pb, T), args.cpu_seconds)
    return result


# ------------------------------------------------------ MLA latent cache
def run_mla(args, rank, world, local):
    """A step = pgd_mla_append_decode_attention: every sequence's newest
    latent row appended, then every head attends over its sequence's latent
    cache (and cut units are merged); bytes = each cached token's 576 bf16
    values once."""
    import torch

    import __graft_entry__
    import paged_gqa_decode_kv_gb300 as pgd
    from paged_gqa_decode_kv_gb300 import inputs

    __graft_entry__.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    name = args.workload if args.workload in inputs.MLA_WORKLOADS else "mla128_batch16_ctx8192"
    mb = inputs.make_mla_workload(name, device=dev, append=True)
    B, H = mb.batch, mb.heads
    nbytes = inputs.mla_bytes_read(mb)
    flops = int(mb.context_lens.sum().item()) * H * (inputs.MLA_D + inputs.MLA_DV) * 2
    pool_b = mb.cache.numel() * 2
    n_pools = 1 if pool_b > 2 * L2_BYTES else -(-2 * L2_BYTES // pool_b)
    pools = [mb.cache] + [mb.cache.clone() for _ in range(n_pools - 1)]
    ws = torch.empty(max(256, pgd.mla_workspace_size(B, H, args.splits)), dtype=torch.uint8,
                     device=dev)
    out = torch.empty((B, H, inputs.MLA_DV), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()
    it = [0]

    def next_pool():
        c = pools[it[0] % n_pools]
        it[0] += 1
        return c

    def attend(c, q_=None, out_=None, lens=None):
        pgd.mla_decode_attention(out if out_ is None else out_, mb.q if q_ is None else q_, c,
                                 mb.block_tables, mb.context_lens if lens is None else lens,
                                 mb.scale, num_splits=args.splits, workspace=ws, stream=stream)

    def step():
        c = next_pool()
        pgd.mla_append_decode_attention(out, mb.q, mb.c_new, c, mb.block_tables,
                                        mb.context_lens, mb.scale, num_splits=args.splits,
                                        workspace=ws, stream=stream)

    gpu_uuid = "GPU-" + str(torch.cuda.get_device_properties(local).uuid)
    sampler = ClockSampler(gpu_uuid)
    sampler.start()
    nvml = NvmlClocks(gpu_uuid)
    nvml.start()
    time.sleep(0.3)
    t_wall0 = time.time()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    flags = pgd.device_errors(clear=True, stream=stream)
    if flags:
        raise RuntimeError("device error word %d after warm-up" % flags)
    K = args.steps
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t_timed0 = time.time()
    e0.record(stream)
    for _ in range(K):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    t_timed1 = time.time()
    barrier(world)
    ev_a = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev_b = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for i in range(K):
        c = next_pool()
        ev_a[i].record(stream)
        attend(c)
        ev_b[i].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    t_wall1 = time.time()
    time.sleep(0.25)
    sampler.stop()
    nvml.stop()
    elapsed_ms = e0.elapsed_time(e1)
    attn_all = [a.elapsed_time(b) for a, b in zip(ev_a, ev_b)]
    attn_ms = statistics.fmean(attn_all)
    attn_med = statistics.median(attn_all)
    flags = pgd.device_errors(clear=True, stream=stream)
    if flags:
        raise RuntimeError("device error word %d after the timed steps" % flags)
    max_ms = max_over_ranks(elapsed_ms, world)
    value = sum_over_ranks(nbytes * K, world) / (max_ms / 1e3) / 1e9

    # end to end through pgd_mla_step: pinned host queries (copied), new rows
    # and context lengths (read in place) in, latent outputs (written in
    # place) back
    q_h, cn_h = mb.q.cpu().pin_memory(), mb.c_new.cpu().pin_memory()
    cl_h = mb.context_lens.cpu().pin_memory()
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    q_d, cn_d = torch.empty_like(mb.q), torch.empty_like(mb.c_new)
    cl_d = torch.empty_like(mb.context_lens)

    def e2e_step():
        c = next_pool()
        pgd.mla_step(out_h, q_h, cn_h, cl_h, out, q_d, cn_d, cl_d, c, mb.block_tables, mb.scale,
                     args.splits, ws, stream=stream)

    for _ in range(args.warmup):
        e2e_step()
    torch.cuda.synchronize()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(K):
        e2e_step()
    f1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(f0.elapsed_time(f1), world)
    ro_best, ro_rec = read_only_peak(dev, stream)
    peak, peak_kind = hbm_peak()
    achieved = nbytes / (attn_ms / 1e3) / 1e9
    parts = args.splits if args.splits > 0 else max(1, min(
        64, torch.cuda.get_device_properties(local).multi_processor_count // (B * -(-H // 64))))
    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(max_ms / K, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "accumulate": "f32",
        "data": "synthetic (seeded N(0,1) bf16 latent rows and absorbed queries, random block "
                "tables)",
        "config": {"workload": name, "batch": B, "heads": H, "context": int(mb.context_lens[0]),
                   "latent": "576 bf16 per token (512 latent + 64 RoPE key), 512-d output",
                   "block_size": mb.block_size, "parts": parts,
                   "l2": ("latent pool %.0f MB, %d copies rotated (%.0f MB > 2 x L2), no flush"
                          % (pool_b / 1e6, n_pools, n_pools * pool_b / 1e6))},
        "kv_bytes_per_step": nbytes,
        "seq_layer_steps_per_s": round(sum_over_ranks(B * K, world) / (max_ms / 1e3), 1),
        "pct_of_hbm_peak": {"nominal_8tbs": round(100 * value / world / NOMINAL_HBM_GBS, 2),
                            peak_kind: round(100 * value / world / peak, 2),
                            "read_only": round(100 * value / world / ro_best, 2)},
        "read_only_stream": dict(ro_rec, gbs=ro_best),
        "roofline": {"bound": "hbm", "kernel": "pgd::mla::mla_attention_kernel<%d> (tcgen05)"
                     % mb.block_size, "achieved": round(achieved, 2), "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": profiled_mla_traffic(name) if args.splits == 0 else None,
                     "launch_ms": round(attn_ms, 5), "launch_ms_median": round(attn_med, 5),
                     "bytes_per_launch": nbytes,
                     "frac_of_read_only": round(achieved / ro_best, 4),
                     "tflops_achieved": round(flops / (attn_ms / 1e3) / 1e12, 2),
                     "flop_per_byte": round(flops / nbytes, 1)},
        "e2e": {"value": round(sum_over_ranks(nbytes * K, world) / (e2e_ms / 1e3) / 1e9, 2),
                "unit": "GB/s",
                "h2d_bytes_per_step": q_h.numel() * 2 + cn_h.numel() * 2 + cl_h.numel() * 4,
                "d2h_bytes_per_step": out_h.numel() * 2, "ms_per_step": round(e2e_ms / K, 5),
                "path": "pgd_mla_step (host buffers; q copied, the rest in place)"},
        # latent append, attention, merge of the parts
        "gpu_launches": (2 + (1 if parts > 1 else 0)) * K,
        "clocks": clocks_record(sampler, nvml, t_wall0, t_wall1, t_timed0, t_timed1),
        "gpu": torch.cuda.get_device_name(local),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        q_c, c_c = mb.q.cpu(), mb.cache.cpu()
        t_c, l_c = mb.block_tables.cpu(), mb.context_lens.cpu()
        n = 1
        t0 = time.perf_counter()
        oracle.mla_attention(q_c[:n], c_c, t_c[:n], l_c[:n], mb.scale)
        dt = time.perf_counter() - t0
        total_t, total_b, calls = dt, int(l_c[:n].sum()) * inputs.MLA_D * 2, 1
        while total_t < args.cpu_seconds and calls < 64:
            t0 = time.perf_counter()
            oracle.mla_attention(q_c[:n], c_c, t_c[:n], l_c[:n], mb.scale)
            total_t += time.perf_counter() - t0
            total_b += int(l_c[:n].sum()) * inputs.MLA_D * 2
            calls += 1
        result["cpu_baseline"] = {
            "value": round(total_b / total_t / 1e9, 4), "unit": "GB/s",
            "cores": oracle.threads_used(0, n * H), "kind": "oracle",
            "sample": "float64 oracle latent attention over the first sequence (%d heads, %d "
                      "tokens), %d call(s), %.1f s" % (H, int(l_c[0]), calls, total_t)}
    return result


# --------------------------------------------------------- reference arm
def run_reference(args):
    """The oracle, as it stands, on the host cores: each step a bounded sample
    (the first n sequences) of the same workload."""
    import oracle
    from paged_gqa_decode_kv_gb300 import inputs

    pb = inputs.make_workload(args.workload, device="cpu", append=False, kv_format=args.kv)
    host = host_copy(pb)
    B = pb.batch
    # calibrate: one sequence, then size the sample so the run stays within ~2 minutes
    dt1, _ = oracle_sample(host, 1)
    per_step_budget = 120.0 / max(1, args.steps + args.warmup)
    n_seq = int(max(1, min(B, per_step_budget / max(dt1, 1e-6))))
    for _ in range(args.warmup):
        oracle_sample(host, n_seq)
    t_total, b_total = 0.0, 0
    for _ in range(args.steps):
        dt, nb = oracle_sample(host, n_seq)
        t_total += dt
        b_total += nb
    value = b_total / t_total / 1e9
    cores = oracle.threads_used(0, n_seq * pb.n_q)
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(1e3 * t_total / max(1, args.steps), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded %s K/V, N(0,1) bf16 Q, random block tables)"
                % ("E4M3 + per-token scale" if args.kv == "fp8" else "N(0,1) bf16"),
        "config": config_block(pb, args.workload, args.splits, pool_copies(pb)),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                         "kind": "oracle",
                         "sample": "first %d of %d sequences per step (all heads, full context)"
                                   % (n_seq, B)},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    args = parse_args(argv)
    rank, world, local = dist_env()
    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args)), flush=True)
        return 0
    dist_init(world)
    result = run_mla(args, rank, world, local) if args.mla else run_ours(args, rank, world, local)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
