"""Benchmark: attention forward TFLOP/s on GB300 (BF16) and fraction of the
dense BF16 tensor peak.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config mha8k] [--impl ours|reference] [--dynamic]

A step is one exact attention forward (the whole hot path) over the chosen
workload, default the MHA non-causal configuration B4 H16 S8192 d128 (32k
tokens); --config also takes the other fixed-length configurations, the
variable-length batches (varlen32k, varlen32k_nc) and the decode problems
(decode32k, decode_mqa, specdec: split-KV, HBM roofline).  Inputs are synthetic
(seeded N(0,1) bf16) and resident in HBM when
the timed region starts; Q, K, V and O together (514 MiB) are larger than L2,
so no flush is needed between steps.  Prints one JSON line (rank 0).

--impl reference times the fp64 CPU oracle on the host cores on a bounded
sample of the same workload (a deliberately slow baseline, not a target).

Under torchrun (N > 1) every rank runs its own batch of the workload on its
own GPU (weak scaling, no collective on the data path); the timed region is
bracketed by barriers and the slowest rank's time is reported.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOP/s on 1 GB300 (BF16) and % of dense BF16 tensor peak"
METRIC_BWD = "attention bwd TFLOP/s on 1 GB300 (BF16, 2.5x forward flops) and % of dense BF16 tensor peak"
FALLBACK_PEAK_TFLOPS = 1900.0  # burst bf16 of one earlier GB300 measurement
FALLBACK_HBM_GBS = 6800.0      # copy bandwidth of one earlier GB300 measurement
KERNEL_NAME = "fa_fwd_kernel"


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default="mha8k")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--launch-samples", type=int, default=50,
                    help="launches timed one by one after the timed region (mean and median; at least 50; 0 "
                         "skips this pass, for profiler runs)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="CPU-baseline sample budget")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--store-mode", type=int, default=0, choices=(0, 1, 2),
                    help="ablation: the fixed-length epilogue (fa_options.store_mode): 0 chosen by the library, "
                         "1 staged TMA stores, 2 direct stores from registers")
    ap.add_argument("--no-balance", action="store_true",
                    help="ablation: the plain static task order (fa_options.no_balance = 1)")
    ap.add_argument("--stagger", action="store_true",
                    help="ablation: the softmax warpgroups take turns for their exponentials (fa_options.stagger)")
    ap.add_argument("--dynamic", action="store_true",
                    help="fixed-length workloads: assign tasks dynamically (scheduling workspace)")
    ap.add_argument("--pass", dest="pass_", choices=["fwd", "bwd"], default="fwd",
                    help="fwd: the forward (default); bwd: the backward (dQ, dK, dV), flops counted as 2.5x the "
                         "forward's")
    ap.add_argument("--splitkv", type=int, default=0,
                    help="split-KV ranges for fixed-length workloads (decode workloads always split; 0 = auto there)")
    ap.add_argument("--trace", action="store_true",
                    help="fixed-length forward (or, with --pass bwd, backward at head dims 128): run the workload "
                         "once with the kernel's event log (trace build) on the first --trace-ctas CTAs and print the "
                         "interval summary (cycles), with the mean time of the trace build beside the default "
                         "kernel's, instead of timing")
    ap.add_argument("--trace-ctas", type=int, default=8)
    ap.add_argument("--trace-cap", type=int, default=16384)
    ap.add_argument("--trace-out", default=None,
                    help="with --trace: also write the decoded per-CTA event lists (JSON) to this file")
    ap.add_argument("--count-rescales", action="store_true",
                    help="fixed-length forward: run the workload once with the O-rescale counter on and print the "
                         "count, the most the launch could count (warps x K/V blocks after a tile's first) and their "
                         "ratio, instead of timing")
    a = ap.parse_args(argv)
    if a.warmup < 3:
        ap.error("--warmup must be >= 3")
    if a.steps < 1:
        ap.error("--steps must be >= 1")
    return a


# ---------------------------------------------------------------------------
# peaks, clocks, ncu traffic
# ---------------------------------------------------------------------------

def load_peak(key: str = "bf16_tflops"):
    """(value, source): the measured burst bf16 GEMM rate (TFLOP/s) or copy
    bandwidth (hbm_gbs, GB/s), else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d[key]), "measured"
    except Exception:
        return (FALLBACK_PEAK_TFLOPS if key == "bf16_tflops" else FALLBACK_HBM_GBS), "fallback"


class ClockSampler:
    """nvidia-smi samples (SM clock, max clock, throttle reasons) in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, enabled: bool = True):
        self.gpu = gpu_index
        self.enabled = enabled
        self.samples = []
        self.proc = None
        self.thread = None
        self.t0 = self.t1 = None

    def start(self):
        if not self.enabled:
            return
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def mark(self, which):
        if which == "start":
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        return self.summary()

    def summary(self):
        rows = []
        for ts, line in self.samples:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((ts, parts))
        window = [r for r in rows if self.t0 and self.t1 and self.t0 - 0.15 <= r[0] <= self.t1 + 0.15]
        if not window:
            window = rows
        if not window:
            return None
        try:
            mhz = [float(p[1]) for _, p in window]
            mx = max(float(p[2]) for _, p in window)
        except ValueError:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, p in window for i in range(4) if p[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": mx, "reasons": reasons, "samples": len(window),
                "power_w_max": max((float(p[3]) for _, p in window if p[3].replace('.', '', 1).isdigit()),
                                   default=None)}


def kernel_source_hash(which: str = "fwd") -> str:
    """Hash of the sources the forward kernels are built from (the backward's
    and the debug instantiations' files excluded), or with which="bwd" of the
    backward kernels' sources (fa_bwd* and the headers they include); a
    stored ncu figure is valid only for it."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "exact_attention_forward_08_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if which == "bwd":
            if not (name.startswith("fa_bwd") or name in ("ptx.cuh", "fa_kernel.cuh", "fa_schedule.h")):
                continue
        elif name.startswith(("fa_bwd", "fa_dbg_", "fa_var_")):
            continue
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def stored_traffic(config: str):
    """DRAM bytes per launch from the committed ncu summary, if taken on the
    current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", f"fa_fwd_{config}_dram.txt")
    try:
        kv = {}
        with open(path) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("source_hash") != kernel_source_hash():
            return None
        return float(kv["dram_bytes_per_launch"])
    except Exception:
        return None


TC_FLOP_PER_CLK_PER_SM = 8192  # dense bf16 tensor-core rate per SM and clock ("FlashAttention-4 wiki",
                                # "Key observations", observation 1)


def per_launch_times(torch, stream, step, n: int):
    """Mean and median over n launches, each bracketed by its own CUDA events
    on the launching stream (recorded back to back, so the launches still run
    one after the other as in the timed region)."""
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    evs[0].record(stream)
    for i in range(n):
        step()
        evs[i + 1].record(stream)
    torch.cuda.synchronize()
    ms = [evs[i].elapsed_time(evs[i + 1]) for i in range(n)]
    return {"n": n, "mean_ms": round(statistics.fmean(ms), 4), "median_ms": round(statistics.median(ms), 4),
            "min_ms": round(min(ms), 4), "max_ms": round(max(ms), 4)}


def clock_peak(flops: float, ms: float, sms: int, clk):
    """The tensor-core rate implied by the clocks seen during the timed region:
    8192 flop per clock per SM x SMs x the median SM clock under load."""
    if not clk or not clk.get("sm_mhz"):
        return None
    peak = TC_FLOP_PER_CLK_PER_SM * sms * clk["sm_mhz"] * 1e6 / 1e12
    achieved = flops / (ms * 1e-3) / 1e12
    return {"value": round(peak, 1), "unit": "TFLOP/s", "sm_mhz": clk["sm_mhz"], "sms": sms,
            "flop_per_clk_per_sm": TC_FLOP_PER_CLK_PER_SM, "frac": round(achieved / peak, 4)}


# ---------------------------------------------------------------------------
# distributed plumbing (one process per GPU; no data-path collective)
# ---------------------------------------------------------------------------

def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def dist_init(backend: str):
    import torch.distributed as dist
    rank, world, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend, rank=rank, world_size=world)
    return rank, world


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(x: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_batch_seed(base_seed: int, rank: int) -> int:
    """Each rank owns a distinct batch of the workload (distinct inputs)."""
    return base_seed + 1000003 * rank


# ---------------------------------------------------------------------------
# workloads: fixed-length (synthetic.workloads) and varlen (synthetic.varlen_workloads)
# ---------------------------------------------------------------------------

def get_workload(config: str):
    import synthetic
    fixed, varlen, decode = synthetic.workloads(), synthetic.varlen_workloads(), synthetic.decode_workloads()
    for table in (fixed, varlen, decode):
        if config in table:
            return table[config]
    raise SystemExit(f"unknown --config {config!r}; choose from {sorted(fixed) + sorted(varlen) + sorted(decode)}")


def is_decode(config: str) -> bool:
    import synthetic
    return config in synthetic.decode_workloads()


def is_varlen(w) -> bool:
    return hasattr(w, "cu_seqlens_q")


def total_rows(w) -> int:
    return w.total_q * w.heads_q if is_varlen(w) else w.batch * w.seqlen_q * w.heads_q


def oracle_sample(w, q, k, v, n, rng, threads):
    """Run the oracle on n uniformly drawn output rows; returns seconds."""
    import numpy as np
    import oracle
    t0 = time.perf_counter()
    if is_varlen(w):
        rows = np.stack([rng.integers(0, w.total_q, n), rng.integers(0, w.heads_q, n)], axis=1)
        oracle.attn_fwd_varlen(q, k, v, w.cu_seqlens_q, w.cu_seqlens_k, causal=w.causal, scale=w.softmax_scale,
                               rows=rows, threads=threads)
    else:
        rows = rng.integers(0, total_rows(w), size=n, dtype=np.int64)
        oracle.attn_fwd(q, k, v, causal=w.causal, scale=w.softmax_scale, rows=rows, threads=threads)
    return time.perf_counter() - t0


def balance_of(w, sms: int) -> str:
    """The balanced static order the library runs for this workload on `sms` CTAs
    (from its host copy of the schedule)."""
    import exact_attention_forward_08_gb300 as fa
    if is_varlen(w):
        return ""  # varlen batches take their tasks dynamically
    plan = fa.fa_make_plan(w.batch, w.heads_q, w.heads_kv, w.seqlen_q, w.seqlen_k, w.d_qk, w.d_v, int(w.causal))
    n = plan.num_tasks
    fa.fa_plan_set_grid(plan, sms)
    if plan.tail_first < plan.num_tasks:
        r = plan.num_tasks - n
        return f"a partial last wave of {r} tasks runs as {2 * r} key-split tiles"
    if w.causal and plan.mblocks >= 2 and plan.mblocks % 2 == 0 and sms >= 2:
        return "heavy and light m_blocks paired on one CTA"
    return "plain order"


def order_label(w, sms: int, no_balance: bool = False, stagger: bool = False, store_mode: int = 0,
                dynamic: bool = False, splits: int = 1) -> str:
    """The task-order part of the config's task_assignment text, with the
    ablations a run selected (the plain order, the staggered exponentials, a
    forced epilogue mode of the fixed-length kernels)."""
    label = "plain order (ablation)" if no_balance else balance_of(w, sms)
    if stagger and not no_balance:
        label += "; staggered exponentials (ablation)"
    if store_mode and not (dynamic or is_varlen(w) or splits > 1):
        label += {1: "; staged TMA epilogue forced (ablation)", 2: "; direct epilogue forced (ablation)"}[store_mode]
    return label


def config_of(w, world: int, flops: float, dynamic: bool, splits: int = 1, balance: str = "") -> dict:
    assign = "dynamic (task counter)" if dynamic or is_varlen(w) else "static round-robin"
    if balance and not (dynamic or is_varlen(w) or splits > 1):
        assign += "; " + balance
    common = {"heads_q": w.heads_q, "heads_kv": w.heads_kv, "d_qk": w.d_qk, "d_v": w.d_v, "causal": w.causal,
              "flops_per_step_per_gpu": flops,
              "l2": "inputs larger than L2 (Q+K+V+O %.0f MiB per GPU), no flush" % (w.algorithmic_bytes() / 2 ** 20),
              "parallelism": f"weak x{world} (independent batches, no collective)",
              "task_assignment": assign}
    if splits > 1:
        common["split_kv"] = f"{splits} key ranges per task + merge kernel"
    if is_varlen(w):
        return {"workload": f"{w.name}: {w.notes}", "batch_per_gpu": w.batch, "global_batch": w.batch * world,
                "total_tokens": w.total_q, "seq_len": max(w.seqlens_q), **common}
    return {"workload": f"{w.name}: {w.notes}", "batch_per_gpu": w.batch, "global_batch": w.batch * world,
            "seq_len": w.seqlen_q, **common}


# ---------------------------------------------------------------------------
# CPU baseline: the fp64 oracle on a bounded sample of the workload
# ---------------------------------------------------------------------------

def cpu_baseline(w, q, k, v, seconds: float):
    """Time the oracle (as it stands) on uniformly sampled rows of the workload.
    Returns the cpu_baseline object (TFLOP/s counted with the workload's
    nominal flops per row)."""
    import numpy as np
    import oracle

    threads = oracle.default_threads()
    rows_all = total_rows(w)
    per_row = w.flops() / rows_all
    rng = np.random.default_rng(12345)
    n0 = max(threads * 4, 64)
    dt0 = oracle_sample(w, q, k, v, n0, rng, threads)  # calibration
    n = int(min(rows_all, max(n0, n0 * seconds / max(dt0, 1e-3))))
    dt = oracle_sample(w, q, k, v, n, rng, threads)
    return {"value": n * per_row / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{n} of {rows_all} rows of {w.name} drawn uniformly (fp64 C oracle, {threads} threads, "
                      f"{dt:.1f} s)", "seconds": round(dt, 2), "rows": n}


# ---------------------------------------------------------------------------
# end to end: host inputs in, call, results out, pipelined over two slots
# ---------------------------------------------------------------------------

def e2e_pipelined(torch, dev, launch, host_in, dev_in, dev_out, steps: int, warm: int = 3) -> float:
    """Seconds per step of: copy this step's inputs from pinned host memory,
    run `launch(inputs, outputs, stream)`, copy its outputs back to pinned host
    memory.  Two slots of device buffers: the copies of step i+1 (H2D and D2H
    on their own streams) overlap the call of step i, as a pipelined caller
    would run them; every step still moves all of its own bytes.  Slot 0 is
    (dev_in, dev_out); slot 1 is allocated here."""
    ins = [dev_in, [torch.empty_like(t) for t in dev_in]]
    outs = [dev_out, [torch.empty_like(t) for t in dev_out]]
    host_out = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in dev_out] for _ in range(2)]
    comp = torch.cuda.current_stream(dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def run(n):
        for i in range(n):
            k = i % 2
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_done[k])  # the call of step i-2 has read these inputs
                for d_, h_ in zip(ins[k], host_in):
                    d_.copy_(h_, non_blocking=True)
                ev_in[k].record(s_in)
            comp.wait_event(ev_in[k])
            if i >= 2:
                comp.wait_event(ev_out[k])  # step i-2's results have been read back
            launch(ins[k], outs[k], comp.cuda_stream)
            ev_done[k].record(comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[k])
                for h_, d_ in zip(host_out[k], outs[k]):
                    h_.copy_(d_, non_blocking=True)
                ev_out[k].record(s_out)
        torch.cuda.synchronize(dev)

    run(warm)
    barrier()
    t0 = time.perf_counter()
    run(steps)
    return max_over_ranks(time.perf_counter() - t0, dev) / steps


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def run_ours(args):
    import dataclasses

    import numpy as np
    import torch

    import exact_attention_forward_08_gb300 as fa

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init("nccl" if world > 1 else "gloo")
    fa.load_library()
    splits = 1

    w0 = get_workload(args.config)
    w = dataclasses.replace(w0, seed=rank_batch_seed(w0.seed, rank))
    varlen = is_varlen(w)
    qb, kb, vb = w.generate()
    to_t = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    qh, kh, vh = (to_t(a).pin_memory() for a in (qb, kb, vb))
    qd, kd, vd = (t.to(dev) for t in (qh, kh, vh))
    o = torch.empty(w.shapes["o"], dtype=torch.bfloat16, device=dev)
    lse = torch.empty(w.shapes["lse"], dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    scale = w.softmax_scale
    host_inputs, dev_inputs = [qh, kh, vh], [qd, kd, vd]

    if varlen:
        cqh = torch.from_numpy(w.cu_seqlens_q).pin_memory()
        ckh = torch.from_numpy(w.cu_seqlens_k).pin_memory()
        cqd, ckd = cqh.to(dev), ckh.to(dev)
        host_inputs += [cqh, ckh]
        dev_inputs += [cqd, ckd]
        ws_bytes = fa.fa_varlen_workspace_size(w.batch, w.heads_q, w.total_q)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        launches_per_step = 2  # planning kernel + attention kernel

        def launch(ins, outs, stream):
            q_, k_, v_, cq_, ck_ = ins
            rc = fa.fa_fwd_varlen(q_.data_ptr(), k_.data_ptr(), v_.data_ptr(), outs[0].data_ptr(),
                                  outs[1].data_ptr(), cq_.data_ptr(), ck_.data_ptr(), w.batch, w.total_q, w.total_k,
                                  w.heads_q, w.heads_kv, w.d_qk, w.d_v, int(w.causal), scale, ws.data_ptr(),
                                  ws_bytes, stream)
            if rc != 0:
                raise fa.FaError(rc, "fa_fwd_varlen")
    elif is_decode(args.config) or args.splitkv > 0:
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        splits = args.splitkv if args.splitkv > 0 else fa.fa_splitkv_num_splits(
            w.batch, w.heads_q, w.heads_kv, w.seqlen_q, w.seqlen_k, w.d_qk, w.d_v, w.causal, sms)
        ws_bytes = max(fa.fa_splitkv_workspace_size(w.batch, w.heads_q, w.seqlen_q, w.d_v, splits), 16)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        launches_per_step = 2 if splits > 1 else 1  # attention kernel + merge kernel

        def launch(ins, outs, stream):
            rc = fa.fa_fwd_splitkv(ins[0].data_ptr(), ins[1].data_ptr(), ins[2].data_ptr(), outs[0].data_ptr(),
                                   outs[1].data_ptr(), w.batch, w.heads_q, w.heads_kv, w.seqlen_q, w.seqlen_k,
                                   w.d_qk, w.d_v, int(w.causal), scale, splits, ws.data_ptr(), ws_bytes, stream)
            if rc != 0:
                raise fa.FaError(rc, "fa_fwd_splitkv")
    else:
        opts = None
        if args.dynamic:
            ws = torch.zeros(fa.SCHED_WORKSPACE_BYTES, dtype=torch.uint8, device=dev)
            opts = fa.default_options()
            opts.workspace = ws.data_ptr()
        if args.no_balance:
            opts = opts or fa.default_options()
            opts.no_balance = 1
        if args.stagger:
            opts = opts or fa.default_options()
            opts.stagger = 1
        if args.store_mode:
            opts = opts or fa.default_options()
            opts.store_mode = args.store_mode
        launches_per_step = 1

        def launch(ins, outs, stream):
            rc = fa.fa_fwd_ex(ins[0].data_ptr(), ins[1].data_ptr(), ins[2].data_ptr(), outs[0].data_ptr(),
                              outs[1].data_ptr(), w.batch, w.heads_q, w.heads_kv, w.seqlen_q, w.seqlen_k, w.d_qk,
                              w.d_v, int(w.causal), scale, opts, stream)
            if rc != 0:
                raise fa.FaError(rc, "fa_fwd")

    def step():
        launch(dev_inputs, [o, lse], sp)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    code, detail = fa.fa_device_status()
    if code != 0:
        raise fa.FaError(code, f"device status after warm-up {detail}")

    clocks = ClockSampler(local, enabled=not args.no_clocks)
    clocks.start()
    time.sleep(0.3 if clocks.enabled else 0)
    for _ in range(args.warmup):
        step()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(dev)
    clocks.mark("start")
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    clocks.mark("stop")
    barrier()
    ms_total = max_over_ranks(ev0.elapsed_time(ev1), dev)
    # the same launches timed one by one (mean and median), after the timed region
    launches = per_launch_times(torch, stream, step, max(50, args.launch_samples)) if args.launch_samples else None
    clk = clocks.stop()
    code, detail = fa.fa_device_status()
    if code != 0:
        raise fa.FaError(code, f"device status after timed region {detail}")
    ms_step = ms_total / args.steps
    flops = w.flops()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    value = world * flops / (ms_step * 1e-3) / 1e12

    # end to end: pinned host inputs -> device, forward, O and LSE back to host
    e2e_s = e2e_pipelined(torch, dev, launch, host_inputs, dev_inputs, [o, lse], args.e2e_steps)
    h2d = sum(t.numel() * t.element_size() for t in host_inputs)
    d2h = o.numel() * o.element_size() + lse.numel() * lse.element_size()

    hbm_bound = is_decode(args.config)  # K/V read once: bytes, not flops, bound it
    if hbm_bound:
        peak, peak_src = load_peak("hbm_gbs")
        achieved = w.algorithmic_bytes() / (ms_step * 1e-3) / 1e9
    else:
        peak, peak_src = load_peak()
        achieved = flops / (ms_step * 1e-3) / 1e12
    traffic = stored_traffic(args.config) if not args.dynamic else None
    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_of(w, world, flops, args.dynamic, splits,
                            order_label(w, torch.cuda.get_device_properties(dev).multi_processor_count,
                                        args.no_balance, args.stagger, args.store_mode, args.dynamic, splits)),
        "e2e": {"value": round(world * flops / e2e_s / 1e12, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_s * 1e3, 3)},
        "gpu_launches": args.steps * launches_per_step,
        "roofline": {"bound": "hbm" if hbm_bound else "tensor", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "GB/s" if hbm_bound else "TFLOP/s", "frac": round(achieved / peak, 4),
                     "traffic": traffic,
                     "peak_source": f"{peak_src} ({'copy bandwidth' if hbm_bound else 'bf16 dense, burst'})",
                     "algorithmic_bytes": w.algorithmic_bytes(),
                     "clock_peak": None if hbm_bound else clock_peak(flops, ms_step, sms, clk)},
        "launches": launches,
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(w, qb, kb, vb, args.cpu_seconds)
    elif rank == 0:
        result["cpu_baseline"] = None
    return rank, result


# ---------------------------------------------------------------------------
# our arm, backward
# ---------------------------------------------------------------------------

def bwd_cpu_sample(w, q, k, v, g, seconds: float):
    """Time the backward oracle on the first rows of every (batch, head): the
    same key count and heads, fewer query rows (the oracle's cost per query
    row is that of the full problem's).  Returns (TFLOP/s, sample text, s)."""
    import oracle
    threads = oracle.default_threads()

    def run(rows):
        t0 = time.perf_counter()
        oracle.attn_bwd(q[:, :rows], k, v, g[:, :rows], causal=w.causal, scale=w.softmax_scale, threads=threads)
        return time.perf_counter() - t0

    rows = max(1, min(w.seqlen_q, 8))
    dt = run(rows)
    rows = int(max(1, min(w.seqlen_q, rows * seconds / max(dt, 1e-3))))
    dt = run(rows)
    flops = 2.5 * 2.0 * w.batch * w.heads_q * rows * w.seqlen_k * (w.d_qk + w.d_v)
    if w.causal:
        flops /= 2
    text = (f"first {rows} of {w.seqlen_q} query rows of every (batch, head) of {w.name} (fp64 C oracle backward, "
            f"{min(threads, w.batch * w.heads_kv)} threads over batch x key/value heads, {dt:.1f} s)")
    return flops / dt / 1e12, text, dt, min(threads, w.batch * w.heads_kv)


def bwd_cpu_sample_varlen(w, q, k, v, g, seconds: float):
    """The backward oracle on whole sequences of the batch, shortest first,
    until about `seconds` have passed.  Returns (TFLOP/s, sample text, s, cores)."""
    import oracle
    threads = oracle.default_threads()
    order = sorted(range(w.batch), key=lambda b: w.seqlens_q[b] * w.seqlens_k[b])
    cu_q, cu_k = w.cu_seqlens_q, w.cu_seqlens_k
    done, flops, t0 = 0, 0.0, time.perf_counter()
    for b in order:
        q0, q1, k0, k1 = int(cu_q[b]), int(cu_q[b + 1]), int(cu_k[b]), int(cu_k[b + 1])
        if q1 == q0 or k1 == k0:
            continue
        oracle.attn_bwd(q[None, q0:q1], k[None, k0:k1], v[None, k0:k1], g[None, q0:q1], causal=w.causal,
                        scale=w.softmax_scale, threads=threads)
        f = 2.5 * 2.0 * w.heads_q * (q1 - q0) * (k1 - k0) * (w.d_qk + w.d_v)
        flops += f / 2 if w.causal else f
        done += 1
        if time.perf_counter() - t0 > seconds:
            break
    dt = time.perf_counter() - t0
    text = (f"{done} of {w.batch} sequences of {w.name}, shortest first (fp64 C oracle backward, {threads} threads, "
            f"{dt:.1f} s)")
    return flops / dt / 1e12, text, dt, threads


def run_ours_bwd(args):
    import dataclasses

    import numpy as np
    import torch

    import exact_attention_forward_08_gb300 as fa
    import synthetic

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init("nccl" if world > 1 else "gloo")
    fa.load_library()
    w0 = get_workload(args.config)
    if is_decode(args.config):
        raise SystemExit("--pass bwd takes fixed-length or variable-length workloads")
    varlen = is_varlen(w0)
    w = dataclasses.replace(w0, seed=rank_batch_seed(w0.seed, rank))
    qb, kb, vb = w.generate()
    gb = synthetic.normal_bf16(w.shapes["o"], w.seed, 7)
    to_t = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    qh, kh, vh, gh = (to_t(a).pin_memory() for a in (qb, kb, vb, gb))
    qd, kd, vd, gd = (t.to(dev) for t in (qh, kh, vh, gh))
    if varlen:
        cq = torch.tensor(w.cu_seqlens_q, dtype=torch.int32, device=dev)
        ck = torch.tensor(w.cu_seqlens_k, dtype=torch.int32, device=dev)
        o, lse = fa.attention_forward_varlen(qd, kd, vd, cq, ck, causal=w.causal, scale=w.softmax_scale)
        ws_bytes = fa.fa_bwd_varlen_workspace_size(w.batch, w.heads_q, w.heads_kv, w.total_q, w.total_k)
    else:
        o, lse = fa.attention_forward(qd, kd, vd, causal=w.causal, scale=w.softmax_scale)
        ws_bytes = fa.fa_bwd_workspace_size(w.batch, w.heads_q, w.seqlen_q)
    oh, lh = o.cpu().pin_memory(), lse.cpu().pin_memory()
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    sp = torch.cuda.current_stream(dev).cuda_stream
    scale = w.softmax_scale

    bopts = None
    if args.no_balance:
        bopts = fa.default_options()
        bopts.no_balance = 1

    def launch(ins, outs, stream):
        q_, k_, v_, o_, l_, g_ = ins
        if varlen:
            rc = fa.fa_bwd_varlen(q_.data_ptr(), k_.data_ptr(), v_.data_ptr(), o_.data_ptr(), l_.data_ptr(),
                                  g_.data_ptr(), outs[0].data_ptr(), outs[1].data_ptr(), outs[2].data_ptr(),
                                  cq.data_ptr(), ck.data_ptr(), w.batch, w.total_q, w.total_k, w.heads_q, w.heads_kv,
                                  w.d_qk, w.d_v, int(w.causal), scale, ws.data_ptr(), ws_bytes, stream)
        else:
            rc = fa.fa_bwd(q_.data_ptr(), k_.data_ptr(), v_.data_ptr(), o_.data_ptr(), l_.data_ptr(), g_.data_ptr(),
                           outs[0].data_ptr(), outs[1].data_ptr(), outs[2].data_ptr(), w.batch, w.heads_q, w.heads_kv,
                           w.seqlen_q, w.seqlen_k, w.d_qk, w.d_v, int(w.causal), scale, ws.data_ptr(), ws_bytes,
                           stream, bopts)
        if rc != 0:
            raise fa.FaError(rc, "fa_bwd")

    def step():
        launch([qd, kd, vd, o, lse, gd], [dq, dk, dv], sp)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    code, detail = fa.fa_device_status()
    if code != 0:
        raise fa.FaError(code, f"device status after warm-up {detail}")
    clocks = ClockSampler(local, enabled=not args.no_clocks)
    clocks.start()
    time.sleep(0.3 if clocks.enabled else 0)
    for _ in range(args.warmup):
        step()
    stream = torch.cuda.current_stream(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(dev)
    clocks.mark("start")
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    clocks.mark("stop")
    barrier()
    ms_total = max_over_ranks(ev0.elapsed_time(ev1), dev)
    # the same launches timed one by one (mean and median), after the timed region
    launches = per_launch_times(torch, stream, step, max(50, args.launch_samples)) if args.launch_samples else None
    clk = clocks.stop()
    code, detail = fa.fa_device_status()
    if code != 0:
        raise fa.FaError(code, f"device status after timed region {detail}")
    ms_step = ms_total / args.steps
    flops = 2.5 * w.flops()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    value = world * flops / (ms_step * 1e-3) / 1e12

    # end to end: the backward's inputs in, the three gradients out
    host_in, dev_in = [qh, kh, vh, oh, lh, gh], [qd, kd, vd, o, lse, gd]
    e2e_s = e2e_pipelined(torch, dev, launch, host_in, dev_in, [dq, dk, dv], args.e2e_steps)
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in (dq, dk, dv))
    peak, peak_src = load_peak()
    achieved = flops / (ms_step * 1e-3) / 1e12
    if varlen:
        order = "sequences longest first (planning kernel), static round-robin"
    else:
        blocks_even = -(-w.seqlen_q // 128) % 2 == 0 and -(-w.seqlen_k // 128) % 2 == 0
        order = ("plain order (ablation)" if args.no_balance else
                 ("heavy and light blocks paired on one CTA" if w.causal and blocks_even else "plain order"))
    cfg = config_of(w, world, flops, False, 1, order)
    cfg["pass"] = "backward (dQ, dK, dV; flops = 2.5x forward, 5 GEMMs; the kernels run 7)"
    result = {
        "metric": METRIC_BWD, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": cfg,
        "e2e": {"value": round(world * flops / e2e_s / 1e12, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_s * 1e3, 3)},
        # row preparation, dK/dV kernel, dQ kernel (and the planning kernel for varlen)
        "gpu_launches": args.steps * (4 if varlen else 3),
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "traffic": None,
                     "peak_source": f"{peak_src} (bf16 dense, burst)", "algorithmic_flops": flops,
                     "clock_peak": clock_peak(flops, ms_step, sms, clk)},
        "launches": launches,
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v_, text, dt, cores = (bwd_cpu_sample_varlen if varlen else bwd_cpu_sample)(w, qb, kb, vb, gb,
                                                                                  args.cpu_seconds)
        result["cpu_baseline"] = {"value": v_, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": text,
                                  "seconds": round(dt, 2)}
    elif rank == 0:
        result["cpu_baseline"] = None
    return rank, result


# ---------------------------------------------------------------------------
# reference arm: the fp64 oracle on the host cores
# ---------------------------------------------------------------------------

def run_reference(args):
    """Each step runs the oracle (as it stands) on a bounded uniform sample of
    the workload's rows; the sample size keeps the whole run to about two
    minutes.  Rank 0 alone runs; other ranks exit without work."""
    import numpy as np
    import oracle

    rank, world, _ = dist_env()
    if rank != 0:
        return rank, None
    w = get_workload(args.config)
    q, k, v = w.generate()
    threads = oracle.default_threads()
    if args.pass_ == "bwd":
        return rank, run_reference_bwd(args, w, q, k, v)
    rows_all = total_rows(w)
    per_row = w.flops() / rows_all
    rng = np.random.default_rng(777)

    n_cal = max(4 * threads, 64)
    rate = n_cal / max(oracle_sample(w, q, k, v, n_cal, rng, threads), 1e-3)  # rows per second
    per_step_s = min(10.0, 120.0 / (args.steps + args.warmup))
    n = int(max(threads, min(rows_all, rate * per_step_s)))
    for _ in range(args.warmup):
        oracle_sample(w, q, k, v, n, rng, threads)
    times = [oracle_sample(w, q, k, v, n, rng, threads) for _ in range(args.steps)]
    s_step = sum(times) / len(times)
    value = n * per_row / s_step / 1e12
    sample = (f"{n} of {rows_all} rows of {w.name} per step, drawn uniformly; fp64 C oracle on {threads} "
              f"host threads")
    cfg = config_of(w, 1, w.flops(), False)
    cfg["rows_per_step"] = n
    result = {
        "metric": METRIC, "impl": "reference", "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(s_step * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": cfg,
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    return rank, result


def run_reference_bwd(args, w, q, k, v):
    """The backward oracle, each step on the first rows of every (batch, head)
    (bwd_cpu_sample; whole sequences for a variable-length batch), sized so
    the whole run stays near two minutes."""
    import synthetic
    sample = bwd_cpu_sample_varlen if is_varlen(w) else bwd_cpu_sample
    g = synthetic.normal_bf16(w.shapes["o"], w.seed, 7)
    per_step = min(10.0, 120.0 / (args.steps + args.warmup))
    for _ in range(args.warmup):
        sample(w, q, k, v, g, per_step)
    runs = [sample(w, q, k, v, g, per_step) for _ in range(args.steps)]
    value = sum(r[0] for r in runs) / len(runs)
    cfg = config_of(w, 1, 2.5 * w.flops(), False)
    cfg["pass"] = "backward (flops = 2.5x forward)"
    return {
        "metric": METRIC_BWD, "impl": "reference", "value": value, "unit": "TFLOP/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(sum(r[2] for r in runs) / len(runs) * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": cfg,
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": runs[0][3], "kind": "oracle",
                         "sample": runs[0][1]},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def trace_run(args) -> dict:
    """One forward launch of a fixed-length workload with the event log on
    (fa_options.trace) and the interval summary of exact_attention_forward_08_gb300.trace."""
    import numpy as np
    import torch
    import exact_attention_forward_08_gb300 as fa
    from exact_attention_forward_08_gb300 import trace as tr
    w = get_workload(args.config)
    if is_varlen(w) or is_decode(args.config):
        raise SystemExit("--trace takes a fixed-length --config")
    fa.load_library()
    to_dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    q, k, v = (to_dev(a) for a in w.generate())
    o = torch.empty(w.shapes["o"], dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(w.shapes["lse"], dtype=torch.float32, device="cuda")
    words = tr.trace_words(args.trace_ctas, args.trace_cap)
    buf = torch.zeros(words, dtype=torch.int64, device="cuda")
    topts = fa.default_options()
    topts.trace = buf.data_ptr()
    topts.trace_ctas = args.trace_ctas
    topts.trace_cap = args.trace_cap
    stream = torch.cuda.current_stream()

    def launch(opts):
        rc = fa.fa_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), w.batch, w.heads_q,
                          w.heads_kv, w.seqlen_q, w.seqlen_k, w.d_qk, w.d_v, int(w.causal), w.softmax_scale, opts,
                          stream.cuda_stream)
        if rc != 0:
            raise fa.FaError(rc, "fa_fwd_ex")

    def mean_ms(opts, n=10):
        for _ in range(3):
            launch(opts)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            launch(opts)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    base_ms = mean_ms(None)
    trace_ms = mean_ms(topts)
    buf.zero_()
    launch(topts)
    torch.cuda.synchronize()
    code, detail = fa.fa_device_status()
    if code != 0:
        raise SystemExit(f"device status {code} {detail}")
    host = buf.cpu().numpy().view(np.uint64)
    ctas = tr.decode(host, args.trace_ctas, args.trace_cap)
    dropped = sum(max(0, n - args.trace_cap) for c in ctas for n in c["_counts"].values())
    if args.trace_out:
        with open(args.trace_out, "w") as f:
            json.dump(ctas, f)
    return {"config": args.config, "workload": f"{w.name}: {w.notes}", "trace_ctas": args.trace_ctas,
            "records_dropped": dropped, "kernel_ms_default": round(base_ms, 4),
            "kernel_ms_trace_build": round(trace_ms, 4), "unit": "SM clock cycles",
            "summary": tr.summarize(ctas)}


def trace_run_bwd(args) -> dict:
    """One backward call (dK/dV and dQ kernels) of a fixed-length (128, 128)
    workload with the event log on, and the interval summary of each kernel."""
    import numpy as np
    import torch
    import exact_attention_forward_08_gb300 as fa
    import synthetic
    from exact_attention_forward_08_gb300 import trace as tr
    w = get_workload(args.config)
    if is_varlen(w) or is_decode(args.config):
        raise SystemExit("--trace takes a fixed-length --config")
    fa.load_library()
    to_dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    q, k, v = (to_dev(a) for a in w.generate())
    g = to_dev(synthetic.normal_bf16(w.shapes["o"], w.seed, 7))
    o, lse = fa.attention_forward(q, k, v, causal=w.causal, scale=w.softmax_scale)
    words = tr.trace_words(args.trace_ctas, args.trace_cap)
    buf = torch.zeros(2 * words, dtype=torch.int64, device="cuda")
    topts = fa.default_options()
    topts.trace = buf.data_ptr()
    topts.trace_ctas = args.trace_ctas
    topts.trace_cap = args.trace_cap

    def mean_ms(opts, n=5):
        for _ in range(2):
            fa.attention_backward(q, k, v, o, lse, g, causal=w.causal, scale=w.softmax_scale, options=opts)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n):
            fa.attention_backward(q, k, v, o, lse, g, causal=w.causal, scale=w.softmax_scale, options=opts)
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    base_ms = mean_ms(None)
    trace_ms = mean_ms(topts)
    buf.zero_()
    fa.attention_backward(q, k, v, o, lse, g, causal=w.causal, scale=w.softmax_scale, options=topts)
    torch.cuda.synchronize()
    code, detail = fa.fa_device_status()
    if code != 0:
        raise SystemExit(f"device status {code} {detail}")
    host = buf.cpu().numpy().view(np.uint64)
    out = {"config": args.config, "pass": "bwd", "workload": f"{w.name}: {w.notes}", "trace_ctas": args.trace_ctas,
           "call_ms_default": round(base_ms, 4), "call_ms_trace_build": round(trace_ms, 4),
           "unit": "SM clock cycles"}
    raw = {}
    for kind, name in ((0, "dkdv"), (1, "dq")):
        ctas = tr.decode(host[kind * words:(kind + 1) * words], args.trace_ctas, args.trace_cap)
        raw[name] = ctas
        out[f"{name}_records_dropped"] = sum(max(0, n - args.trace_cap) for c in ctas for n in c["_counts"].values())
        out[f"{name}_summary"] = tr.summarize_bwd(ctas)
    if args.trace_out:
        with open(args.trace_out, "w") as f:
            json.dump(raw, f)
    return out


def count_rescales(args) -> dict:
    """One forward launch of a fixed-length workload with the correction warps'
    O-rescale counter on (fa_options.debug_flags bit 1), in the checking build
    (bit 2), whose arithmetic and rescale decisions are the default kernel's."""
    import numpy as np
    import torch
    import exact_attention_forward_08_gb300 as fa
    w = get_workload(args.config)
    if is_varlen(w) or is_decode(args.config):
        raise SystemExit("--count-rescales takes a fixed-length --config")
    fa.load_library()
    to_dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    q, k, v = (to_dev(a) for a in w.generate())
    opts = fa.default_options()
    opts.debug_flags = fa.DEBUG_COUNT_RESCALE | fa.DEBUG_CHECKS
    fa.fa_device_status()
    fa.attention_forward(q, k, v, causal=w.causal, scale=w.softmax_scale, options=opts)
    n = fa.fa_debug_rescale_count()
    code = fa.fa_device_status()[0]
    if code != 0:
        raise SystemExit(f"device status {code}")
    plan = fa.fa_make_plan(w.batch, w.heads_q, w.heads_kv, w.seqlen_q, w.seqlen_k, w.d_qk, w.d_v, int(w.causal))
    # the order the launch ran (key-split tasks count each half's blocks after its first)
    fa.fa_plan_set_grid(plan, torch.cuda.get_device_properties(0).multi_processor_count)
    total = 0
    for t in range(plan.num_tasks):
        task = fa.fa_plan_task(plan, t)
        total += sum(4 * max(0, task.n_blocks[s] - 1) for s in range(2))
    return {"config": args.config, "rescales": n, "opportunities": total,
            "rate": (n / total) if total else 0.0,
            "unit": "warps of 32 rows x K/V blocks after the first whose O was rescaled"}


def main(argv=None):
    args = parse_args(argv)
    if args.count_rescales:
        print(json.dumps(count_rescales(args)), flush=True)
        return 0
    if args.trace:
        print(json.dumps(trace_run_bwd(args) if args.pass_ == "bwd" else trace_run(args)), flush=True)
        return 0
    if args.impl == "reference":
        runner = run_reference
    else:
        runner = run_ours_bwd if args.pass_ == "bwd" else run_ours
    rank, result = runner(args)
    if rank == 0 and result is not None:
        print(json.dumps(result), flush=True)
    try:
        import torch.distributed as dist
        if dist.is_available() and dist.is_initialized():
            dist.destroy_process_group()
    except Exception:
        pass
    return 0


if __name__ == "__main__":
    sys.exit(main())
