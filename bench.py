"""Benchmark of the LampAttention forward pass on GB300.

A step is one lamp_attn_fwd call over the whole workload (pre-pass + fused
kernel, mask bytes and counters collected), inputs resident in HBM.  Default
workload: the Qwen3-8B attention shape (B4, N4096, 32 query / 8 KV heads,
d128, causal, bf16) at tau = 2^-1, delta = 2^-8, with seeded synthetic
inputs (outlier channels + sink key).  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl lamp|reference]

--impl reference times the CPU oracle (float64 NumPy, all host cores) on a
bounded sample of query tiles of the same workload.
"""
from __future__ import annotations

import argparse
import json
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from mixed_precision_flashattention_gb300 import synth  # noqa: E402

METRIC = "attn fwd TFLOP/s & % FP8 peak, Qwen3-8B shape 4k ctx; 16-bit sub-block frac"
FLUSH_BYTES = 256 << 20  # > 129 MB L2


# ---------------------------------------------------------------- CPU oracle leg
def _oracle_task(args):
    qv, kv, vv, tiles, mask, window, delta, tau, pv, qk = args
    import oracle
    t0 = time.perf_counter()
    oracle.lamp_forward(qv, kv, vv, mask=mask, window=window, delta=delta, tau=tau, tiles=tiles, pv=pv, qk=qk)
    return time.perf_counter() - t0


def _tile_flops(w, i):
    """Algorithmic FLOPs of query tile i (64 rows) of one head."""
    n = w.seqlen
    rows = np.arange(64 * i, min(64 * i + 64, n))
    if w.mask == "none":
        vis = np.full(rows.shape, n)
    elif w.mask == "causal":
        vis = rows + 1
    else:
        vis = np.minimum(rows + 1, w.window)
    return 4.0 * w.head_dim * float(vis.sum())


def _head_values(w, x, b, h):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x[b:b + 1, :, h:h + 1]))
    return (t.to(torch.bfloat16) if w.dtype == "bf16" else t).double().numpy()


def cpu_sample_tasks(w, q, k, v, delta, tau, wall_budget_s, ncores, seed=0, pv="fp16", qk="exact"):
    """Bounded sample of the workload for the CPU oracle: random
    (batch, head, query-tile) triples until the estimated wall time on
    ``ncores`` workers reaches ``wall_budget_s``.  One task per head."""
    T = (w.seqlen + 63) // 64
    grp = w.heads_q // w.heads_kv
    probe = (_head_values(w, q, 0, 0), _head_values(w, k, 0, 0), _head_values(w, v, 0, 0),
             [(0, 0, T - 1)], w.mask, w.window, delta, tau, pv, qk)
    t_long = _oracle_task(probe)  # seconds for the longest query tile
    rng = np.random.default_rng(seed)
    picks, est, n = {}, 0.0, 0
    cap = min(8192, w.batch * w.heads_q * T)  # a small workload is sampled whole
    while est < wall_budget_s * ncores and n < cap:
        b, h, i = int(rng.integers(w.batch)), int(rng.integers(w.heads_q)), int(rng.integers(T))
        if i in picks.get((b, h), ()):
            continue
        picks.setdefault((b, h), []).append(i)
        n += 1
        est += t_long * _tile_flops(w, i) / _tile_flops(w, T - 1)
    tasks, flops = [], 0.0
    for (b, h), tiles in picks.items():
        g = h // grp
        tasks.append((_head_values(w, q, b, h), _head_values(w, k, b, g), _head_values(w, v, b, g),
                      [(0, 0, i) for i in sorted(tiles)], w.mask, w.window, delta, tau, pv, qk))
        flops += sum(_tile_flops(w, i) for i in tiles)
    return tasks, flops


def run_cpu_oracle(pool, tasks):
    t0 = time.perf_counter()
    list(pool.imap_unordered(_oracle_task, tasks))
    return time.perf_counter() - t0


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock and throttle-reason samples (every 20 ms) with their
    timestamps; only the samples inside the timed region are reported."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0):
        self.index = index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"lamp_bench_clocks_{os.getpid()}.csv")
        self.t0 = self.t1 = None

    def start(self):
        """Start sampling; returns once the first sample is written (or after 5 s)."""
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        deadline = time.time() + 5.0
        while time.time() < deadline and self.proc.poll() is None:
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.01)

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    @staticmethod
    def _when(stamp):
        import datetime
        for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
            try:
                return datetime.datetime.strptime(stamp, fmt).timestamp()
            except ValueError:
                pass
        return None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        self.proc.wait(timeout=10)
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 10:
                rows.append(parts)
        os.remove(self.path)
        if not rows:
            return None
        inside = rows
        if self.t0 is not None and self.t1 is not None:
            stamped = [(self._when(r[0]), r) for r in rows]
            inside = [r for t, r in stamped if t is not None and self.t0 <= t <= self.t1]
            if not inside:  # region shorter than the sampling period: the samples around it
                before = [r for t, r in stamped if t is not None and t <= self.t1]
                after = [r for t, r in stamped if t is not None and t > self.t1]
                inside = before[-1:] + after[:1]
        sm = [float(r[2]) for r in inside if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in inside if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[j] for r in inside for j in range(4) if r[6 + j].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside)}


KERNEL_SOURCES = ["mixed_precision_flashattention_gb300/csrc/lamp_fwd.cu",
                  "mixed_precision_flashattention_gb300/csrc/lamp_common.cuh",
                  "mixed_precision_flashattention_gb300/csrc/lamp_ptx.cuh"]


def kernel_source_sha() -> str:
    """Hash of the fused kernel's code: comments and blank lines do not count
    (an edit of a comment leaves the compiled kernel, and so a capture of it,
    unchanged)."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        src = open(os.path.join(ROOT, f), encoding="utf-8").read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for line in src.splitlines():
            line = line.split("//", 1)[0].strip()
            if line:
                h.update(line.encode() + b"\n")
    return h.hexdigest()[:16]


def _capture(workload: str, mode: str = "default"):
    """The committed ncu capture of one fused-kernel launch, if it was taken
    on this workload and kernel mode with the current kernel source (else
    None)."""
    path = os.path.join(ROOT, "profiles", "lamp_fwd_traffic.json")
    if not os.path.exists(path):
        return None
    d = json.load(open(path))
    if d.get("workload") != workload or d.get("source_sha") != kernel_source_sha() or d.get("mode", "default") != mode:
        return None
    return d


def _traffic(workload: str, mode: str = "default"):
    """DRAM bytes per launch of the fused kernel (committed capture)."""
    d = _capture(workload, mode)
    return None if d is None else float(d["dram_bytes_read"]) + float(d["dram_bytes_write"])


def _issue_roofline(workload: str, ms_main: float, sm_mhz, mode: str = "default"):
    """The fused kernel is bound by instruction issue in its softmax warps:
    the floor its warp-instruction count (committed capture) allows at one
    instruction per clock on each of the 4 schedulers of every SM, at the
    SM clock sampled in the timed region, against the measured time."""
    d = _capture(workload, mode)
    if d is None or "warp_instructions" not in d or not sm_mhz:
        return None
    import torch
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    rate = 4.0 * sms * sm_mhz * 1e6  # warp instructions per second
    floor_ms = float(d["warp_instructions"]) / rate * 1e3
    return {"bound": "issue", "warp_instructions": float(d["warp_instructions"]), "sms": sms,
            "sm_mhz": sm_mhz, "floor_ms": floor_ms, "measured_ms": ms_main, "frac": floor_ms / ms_main}


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    return 1900.0, 1700.0, "fallback"


def qkv_fusion_leg(args, w, lamp, torch, dev, flush, bf16_peak):
    """The QKV projection upstream of the attention, two ways, each step from
    the layer input x [B N, hidden] (seeded, synthetic) to out: (a) cuBLAS
    (torch.matmul) writes y = x W^T, q / k / v are strided views of y, and
    the attention runs with its pre-pass; (b) lamp_qkv_project writes q, k,
    v, the K/V cache and the E4M3 copy of q, and the attention runs on them."""
    hidden = args.qkv_fusion
    B, N, Hq, Hkv, d = w.batch, w.seqlen, w.heads_q, w.heads_kv, w.head_dim
    g = torch.Generator(device=dev).manual_seed(args.seed + 11)
    x = (torch.randn(B * N, hidden, device=dev, generator=g) * 0.5).to(torch.bfloat16)
    wt = (torch.randn((Hq + 2 * Hkv) * d, hidden, device=dev, generator=g) / hidden ** 0.5).to(torch.bfloat16)
    probe = torch.empty((B, N, Hq, d), device=dev, dtype=torch.bfloat16)
    kp = torch.empty((B, N, Hkv, d), device=dev, dtype=torch.bfloat16)
    ws = torch.empty(lamp.workspace_bytes(probe, kp, kp), dtype=torch.uint8, device=dev)
    out = torch.empty_like(probe)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=dev)

    def unfused():
        y = torch.matmul(x, wt.t()).view(B, N, Hq + 2 * Hkv, d)
        lamp.lamp_attn_fwd(y[:, :, :Hq], y[:, :, Hq:Hq + Hkv], y[:, :, Hq + Hkv:], mask=w.mask, window=w.window,
                           delta=args.delta, tau=args.tau, out=out, lse=lse, workspace=ws)

    def fused():
        q, k, v = lamp.qkv_project(x, wt, batch=B, heads_q=Hq, heads_kv=Hkv, head_dim=d, workspace=ws)
        lamp.lamp_attn_fwd(q, k, v, mask=w.mask, window=w.window, delta=args.delta, tau=args.tau, out=out,
                           lse=lse, workspace=ws, kv_prepared=True, q_prepared=True)

    def proj_only_cublas():
        torch.matmul(x, wt.t())

    def proj_only_fused():
        lamp.qkv_project(x, wt, batch=B, heads_q=Hq, heads_kv=Hkv, head_dim=d, workspace=ws)

    def timed(fn, n=10):
        ts = []
        for i in range(n + 3):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            if i >= 3:
                ts.append(a.elapsed_time(b))
        return statistics.median(ts)

    proj_flop = 2.0 * B * N * hidden * (Hq + 2 * Hkv) * d
    t_pc, t_pf = timed(proj_only_cublas), timed(proj_only_fused)
    return {"hidden": hidden, "ms_cublas_prepass_attention": timed(unfused), "ms_fused_projection_attention": timed(fused),
            "ms_projection_cublas": t_pc, "ms_projection_fused": t_pf,
            "projection_tflops_cublas": proj_flop / t_pc / 1e9, "projection_tflops_fused": proj_flop / t_pf / 1e9,
            "projection_fused_frac_of_bf16_peak": proj_flop / t_pf / 1e9 / bf16_peak}


def reduce_over_ranks(ms: float, counters, world: int, device=None):
    """Whole-job figures of a multi-rank run: the slowest rank's step time
    and the counters summed over ranks (every rank holds its own shard).
    One rank: returned unchanged."""
    counters = np.asarray(counters, dtype=np.int64)
    if world <= 1:
        return float(ms), counters
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    c = torch.from_numpy(counters.copy()).to(device)
    dist.all_reduce(c, op=dist.ReduceOp.SUM)
    return float(t.item()), c.cpu().numpy()


# ---------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="lamp", choices=["lamp", "reference"])
    ap.add_argument("--workload", default="qwen3_8b", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--tau", type=float, default=0.5)
    ap.add_argument("--delta", type=float, default=2.0 ** -8)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--generator", default=None, choices=sorted(synth.GENERATORS),
                    help="input generator in place of the workload's own (same shape)")
    ap.add_argument("--pv", default="fp16", choices=["fp16", "fp8"],
                    help="P.V precision of unflagged sub-blocks (fp8: the optional FP8 P.V mode)")
    ap.add_argument("--qkv-fusion", type=int, default=0, metavar="HIDDEN",
                    help="also time the QKV projection upstream of the attention (hidden size HIDDEN, bf16): "
                         "cuBLAS GEMM + pre-pass + attention against lamp_qkv_project + attention on its "
                         "K/V cache (an extra 'qkv_fusion' object)")
    ap.add_argument("--kv-prepared", action="store_true",
                    help="keys and values prepared once (lamp_kv_prepare) before the timed steps: "
                         "each step is the forward call on the prepared K/V cache")
    ap.add_argument("--qk", default="exact", choices=["exact", "chunk32"],
                    help="8-bit logit accumulation (chunk32: rounded after every 32-element chunk of d)")
    ap.add_argument("--parity-tiles", type=int, default=64,
                    help="query tiles of the timed inputs checked against the oracle (0: none)")
    args = ap.parse_args()

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    w = synth.WORKLOADS[args.workload]
    if args.generator is not None and args.generator != w.gen:
        import dataclasses
        w = dataclasses.replace(w, name=f"{w.name}_{args.generator}", gen=args.generator)
    flops = w.flops()
    config = {"workload": w.name, "batch": w.batch, "seqlen": w.seqlen, "heads_q": w.heads_q,
              "heads_kv": w.heads_kv, "head_dim": w.head_dim, "mask": w.mask, "window": w.window,
              "in_dtype": w.dtype, "tau": args.tau, "delta": args.delta,
              "generator": w.gen, "seed": args.seed, "pv": args.pv, "qk": args.qk,
              "kv_prepared": bool(args.kv_prepared)}

    if args.impl == "reference" and rank != 0:
        return  # the oracle arm runs on rank 0 only
    want_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
    want_parity = rank == 0 and args.impl == "lamp" and args.parity_tiles > 0
    pool = None
    ncores = os.cpu_count() or 1
    if args.impl == "reference" or want_cpu or want_parity:
        # spawn the oracle's workers before any CUDA call, one BLAS thread each
        for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[var] = "1"
        pool = mp.get_context("spawn").Pool(ncores)

    # rank r holds its own shard of the job: the workload's shape with seed + r
    q, k, v = synth.make(w, seed=args.seed + rank)
    config["inputs_sha256"] = synth.digest(q, k, v)  # of the generated float arrays
    if world > 1:
        config["shard"] = f"rank r of {world}: its own {w.batch} sequences (seed {args.seed} + r)"

    if args.impl == "reference":
        # about 4 x --cpu-seconds of estimated oracle time over the whole run
        # (the pool's transfers roughly double the estimate)
        tasks, sflops = cpu_sample_tasks(w, q, k, v, args.delta, args.tau,
                                         args.cpu_seconds * 4 / max(1, args.steps + args.warmup), ncores,
                                         pv=args.pv, qk=args.qk)
        for _ in range(args.warmup):
            run_cpu_oracle(pool, tasks)
        times = [run_cpu_oracle(pool, tasks) for _ in range(args.steps)]
        pool.close()
        t = statistics.mean(times)
        val = sflops / t / 1e12
        sample = f"{sum(len(x[3]) for x in tasks)} query tiles (64 rows each, all their keys) of {w.name}"
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config,
            "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": ncores, "kind": "oracle", "sample": sample},
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}))
        return

    import torch
    from mixed_precision_flashattention_gb300 import lamp

    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")
    dev = torch.device("cuda")
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    qd, kd, vd = (torch.from_numpy(x).to(dev).to(dt) for x in (q, k, v))
    B, N, Hq, d = qd.shape
    out = torch.empty_like(qd)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=dev)
    mbytes, cnt = lamp.new_stats(B, Hq, N, device=dev)
    ws = torch.empty(lamp.workspace_bytes(qd, kd, vd, out, pv=args.pv, qk=args.qk), dtype=torch.uint8, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    if args.kv_prepared:  # the K/V cache, once, outside the timed region
        lamp.kv_prepare(kd, vd, ws, pv=args.pv, qk=args.qk)

    def step(evs=None, o=out, l=lse, qq=qd, kk=kd, vv=vd):
        lamp.lamp_attn_fwd(qq, kk, vv, mask=w.mask, window=w.window, delta=args.delta, tau=args.tau,
                           out=o, lse=l, mask_bytes=mbytes, counters=cnt, workspace=ws, stage_events=evs,
                           pv=args.pv, qk=args.qk, kv_prepared=args.kv_prepared)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    c = cnt.cpu().numpy()
    if c[9] != 0:
        raise SystemExit(f"device status {c[9]}")

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    for trio in ev:  # create the handles; the library re-records them in each step
        for e in trio:
            e.record()
    clk = ClockSampler(torch.cuda.current_device())
    clk.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    clk.mark_start()
    for i in range(K):
        flush.zero_()
        step(ev[i])
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk.mark_end()
    t_wall = time.perf_counter() - t_wall
    clocks = clk.stop()
    if want_parity:  # outputs of the last timed step, for the parity check below
        out_h = out.float().cpu().numpy().astype(np.float64)
        lse_h = lse.cpu().numpy().astype(np.float64)
        mask_h = mbytes.cpu().numpy()
    t_step = [ev[i][0].elapsed_time(ev[i][2]) for i in range(K)]
    t_prep = [ev[i][0].elapsed_time(ev[i][1]) for i in range(K)]
    t_main = [ev[i][1].elapsed_time(ev[i][2]) for i in range(K)]
    ms, c = reduce_over_ranks(statistics.mean(t_step), cnt.cpu().numpy(), world, dev)
    pct = np.percentile(np.array(t_step), [10, 50, 90]).tolist()
    # the same steps with L2 left warm (no flush): information only
    warm = []
    for i in range(min(K, 20)):
        step(ev[i])
        warm.append(ev[i])
    torch.cuda.synchronize()
    warm_ms = statistics.median(e[0].elapsed_time(e[2]) for e in warm)
    ms_main = statistics.mean(t_main)

    # end to end through the public call on host buffers: pinned host in,
    # copies pipelined against the computation inside the library, host out
    qh, kh, vh = (x.cpu().pin_memory() for x in (qd, kd, vd))
    oh = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    lh = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    hbuf = torch.empty(lamp.host_buffer_bytes(qh, kh, vh, oh, pv=args.pv, qk=args.qk), dtype=torch.uint8,
                       device=dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_ms = []
    for i in range(max(3, K // 2) + 2):
        torch.cuda.synchronize()
        e0.record()
        lamp.lamp_attn_fwd_host(qh, kh, vh, mask=w.mask, window=w.window, delta=args.delta, tau=args.tau,
                                out=oh, lse=lh, mask_bytes=mbytes, counters=cnt, dev_buffer=hbuf, pv=args.pv,
                                qk=args.qk)
        e1.record()
        torch.cuda.synchronize()
        if i >= 2:
            e2e_ms.append(e0.elapsed_time(e1))
    if int(cnt[9].item()) != 0:
        raise SystemExit(f"device status {int(cnt[9].item())} (host-buffer call)")
    h2d = sum(x.numel() * x.element_size() for x in (qh, kh, vh))
    d2h = oh.numel() * oh.element_size() + lh.numel() * lh.element_size()

    # the tau sweep of the pages' figures (tau = 2^0 .. 2^-5 at this delta)
    # from one detector-only pass, against six forward passes
    sweep_taus = [2.0 ** -i for i in range(6)]
    srec = torch.empty((B, Hq, (N + 63) // 64, (N + 63) // 64), dtype=torch.int32, device=dev)
    sw_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(8)]
    for i in range(3 + len(sw_ev)):
        flush.zero_()
        if i >= 3:
            sw_ev[i - 3][0].record()
        sw_hist, _ = lamp.lamp_tau_sweep(qd, kd, sweep_taus, mask=w.mask, window=w.window, delta=args.delta,
                                         records=srec)
        if i >= 3:
            sw_ev[i - 3][1].record()
    torch.cuda.synchronize()
    sweep_ms = statistics.median(a.elapsed_time(b) for a, b in sw_ev)
    e2e_step, _ = reduce_over_ranks(statistics.mean(e2e_ms), [0], world, dev)  # slowest rank
    sw_hist = sw_hist.cpu().numpy()

    # the kernel mode a committed capture must match
    kmode = "pv_fp8" if args.pv == "fp8" else ("qk_chunk32" if args.qk == "chunk32" else "default")
    bf16_peak, bf16_sus, peak_src = _peaks()
    fp8_peak = 2.0 * bf16_peak  # nominal dense FP8 : BF16 ratio of the part
    achieved = flops / (ms_main * 1e-3) / 1e12
    T = (N + 63) // 64
    nqb = (N + 127) // 128
    kv_steps = 0
    for qb in range(nqb):
        last = min(qb * 128 + 127, N - 1)
        if w.mask == "none":
            kv_steps += T
        elif w.mask == "causal":
            kv_steps += last // 64 + 1
        else:
            kv_steps += last // 64 + 1 - max(0, qb * 128 - w.window + 1) // 64
    kv_steps *= B * Hq
    f_step = 2.0 * 128 * 64 * d  # one MMA product of a 128-row x 64-key step
    f_qk8 = kv_steps * f_step
    f_rec = float(c[10] + c[11]) * f_step  # 16-bit products issued: used, or ahead and not needed
    f_rec_used = float(c[10]) * f_step
    if args.pv == "fp8":  # every step's P8.V8, plus P16.V16 for steps with a flagged sub-block
        f_pv8, f_pv = kv_steps * f_step, float(c[10]) * f_step
    else:
        f_pv8, f_pv = 0.0, kv_steps * f_step
    # tensor-core time of the issued work at the peaks: the fastest this
    # kernel design could run on these inputs if the tensor pipe never idled
    t_tc = ((f_qk8 + f_pv8) / (fp8_peak * 1e12) + (f_pv + f_rec) / (bf16_peak * 1e12))
    res = {
        "metric": METRIC, "value": flops / (ms * 1e-3) / 1e12 * world, "unit": "TFLOP/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp8_e4m3+bf16+fp16", "data": "synthetic",
        "config": {**config, "l2": "flushed between steps (256 MB write), per-step CUDA events"},
        "fp8_peak_frac": flops / (ms * 1e-3) / 1e12 / fp8_peak,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": fp8_peak, "unit": "TFLOP/s",
                     "frac": achieved / fp8_peak, "traffic": _traffic(w.name, kmode),
                     "kernel": "lamp_fwd_kernel", "peak_basis": f"2 x {peak_src} bf16 burst {bf16_peak} (dense FP8:BF16 = 2)",
                     "mixed_tc_time_frac": t_tc / (ms_main * 1e-3),
                     "ceiling_fp8_frac": flops / t_tc / 1e12 / fp8_peak,
                     "issue": _issue_roofline(w.name, ms_main, (clocks or {}).get("sm_mhz"), kmode)},
        "ms_main_kernel": ms_main, "ms_prepass": statistics.mean(t_prep), "wall_s": t_wall,
        "ms_per_step_p10_p50_p90": pct, "ms_per_step_l2_warm": warm_ms,
        "stats": {n: int(c[i]) for i, n in enumerate(lamp.COUNTER_NAMES)},
        "subblock16_frac": float(c[6]) / max(1, c[4]),
        "tiles_0_1_2plus": [float(c[1]) / max(1, c[0]), float(c[2]) / max(1, c[0]), float(c[3]) / max(1, c[0])],
        "tensor_flops_issued": {"qk_fp8": f_qk8, "pv_fp8": f_pv8, "pv_fp16": f_pv, "recompute_bf16": f_rec,
                                "recompute_bf16_used": f_rec_used},
        "e2e": {"value": flops / (e2e_step * 1e-3) / 1e12 * world, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d * world, "d2h_bytes_per_step": d2h * world, "ms_per_step": e2e_step},
        "tau_sweep": {"taus": sweep_taus, "ms": sweep_ms, "forward_ms": ms, "speedup_vs_forward_per_tau":
                      len(sweep_taus) * ms / sweep_ms,
                      "tiles_0_1_2plus": [[float(x) / max(1, hrow[0]) for x in hrow[1:]] for hrow in sw_hist]},
        # pre-pass (+ the V8 copy for the FP8 P.V) + fused kernel per step and rank; with a
        # prepared K/V cache and bf16 q the pre-pass has no work and is not launched
        "gpu_launches": (1 if (args.kv_prepared and w.dtype == "bf16") else
                         (2 if args.kv_prepared else (3 if args.pv == "fp8" else 2))) * K * world,
        "clocks": clocks,
    }
    if args.qkv_fusion and w.dtype == "bf16":
        res["qkv_fusion"] = qkv_fusion_leg(args, w, lamp, torch, dev, flush, bf16_peak)
    if want_cpu:
        tasks, sflops = cpu_sample_tasks(w, q, k, v, args.delta, args.tau, args.cpu_seconds, ncores, pv=args.pv,
                                         qk=args.qk)
        tcpu = run_cpu_oracle(pool, tasks)
        res["cpu_baseline"] = {"value": sflops / tcpu / 1e12, "unit": "TFLOP/s", "cores": ncores, "kind": "oracle",
                               "sample": f"{sum(len(x[3]) for x in tasks)} query tiles of {w.name}, {tcpu:.1f} s"}
    if want_parity:
        from tests import sampled_parity as sp
        tiles = sp.sample_tiles(w.batch, w.heads_q, w.seqlen, args.parity_tiles, seed=args.seed)
        ptasks, pkeys = sp.make_tasks(q, k, v, tiles, bf16=w.dtype == "bf16", heads_q=w.heads_q,
                                      heads_kv=w.heads_kv, mask=w.mask, window=w.window, delta=args.delta,
                                      tau=args.tau, out_dtype=w.dtype, pv=args.pv, qk=args.qk)
        presults = pool.map(sp.oracle_task, ptasks)
        par = sp.compare(presults, pkeys, out_h, lse_h, mask_h, w.dtype, w.seqlen, w.mask, w.window)
        par["sample"] = (f"{par['tiles']} query tiles (64 rows, all their keys) of the last timed step's "
                         f"inputs and outputs, seed {args.seed}")
        res["parity"] = par
    if pool is not None:
        pool.close()
    if rank == 0:
        print(json.dumps(res))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
