#!/usr/bin/env python3
"""Attention forward+backward throughput on one GB300, as TFLOP/s and as a
fraction of the dense-bf16 roofline.

One step = the whole path on one batch already resident in device memory:
fa_fwd, then the backward as its three launches (fa_bwd_prep, fa_bwd_dkdv,
fa_bwd_dq).  FLOPs per the usual convention: forward 4*B*H*N^2*d, backward
2.5x forward, both halved under the causal mask.

Default workload: B=2, H=16, N=8192, d=128, causal, Q/K scaled by 3 (the
large-head-dimension training step); its inputs (4 x 64 MiB) are larger than
L2, so no flush is needed between steps.  A vs-N sweep over the other
workloads (forward, or forward+backward where they have one) follows, each
with an L2 flush between timed iterations.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun every rank runs the same per-GPU workload (weak scaling, no
data-path collective); rank 0 prints one JSON line.
"""
import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from exact_attention_04_gb300.workloads import (WORKLOADS, block_sparse_mask,  # noqa: E402
                                                make_inputs, random_case)

METRIC = "attention fwd/bwd TFLOP/s on 1 GB300 and % of dense-BF16 roofline vs N"
HEADLINE = "large_head_b2_h16_n8192_d128_causal"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
# Every source a kernel's DRAM traffic depends on: its own file, the headers
# it includes, and fa_api.cu (the host planner that sets its schedule).
_COMMON_SOURCES = ["fa_api.cu", "fa_internal.h", "fa_window.cuh", "sm103_ptx.cuh"]
KERNEL_SOURCES = {
    "fa_fwd_kernel": ["fa_fwd.cu"] + _COMMON_SOURCES,
    "bwd_d64_kernel": ["fa_bwd_d64.cu", "fa_bwd_common.cuh"] + _COMMON_SOURCES,
    "bwd_dt_kernel": ["fa_bwd_dt.cu", "fa_bwd_common.cuh"] + _COMMON_SOURCES,
}


def bwd_kernel_names(d):
    """Device names of the backward's main and dQ-conversion kernels: d = 64
    runs the query-row kernel, d = 128 and 256 the transposed-dQ one."""
    return ("bwd_d64_kernel", "bwd_post_kernel") if d == 64 else ("bwd_dt_kernel",
                                                                    "bwd_post_t_kernel")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(WORKLOADS))
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch size (small cases for profiling)")
    ap.add_argument("--fp8", action="store_true",
                    help="time the E4M3 forward (quantiser + FP8 kernel) of the workload instead")
    ap.add_argument("--sweep-only", default=None, metavar="SUBSTR",
                    help="run only the sweep entries whose workload name contains SUBSTR "
                         "(no headline step) and print them as one JSON line")
    return ap.parse_args()


# ------------------------------------------------------------------ distributed plumbing

class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        t = torch.tensor([x], dtype=torch.float64,
                         device="cuda" if torch.cuda.is_available() else "cpu")
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ------------------------------------------------------------------ helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return {k: float(pk[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def source_sha(kernel):
    h = hashlib.sha256()
    for name in KERNEL_SOURCES.get(kernel, []):
        with open(os.path.join(ROOT, "exact_attention_04_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def committed_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if it still
    describes the current source of that kernel on this workload."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            entries = json.load(f)
    except (OSError, ValueError):
        return None
    for e in entries:
        if e.get("kernel") == kernel and e.get("workload") == workload \
                and e.get("source_sha") == source_sha(kernel):
            return e.get("dram_bytes_per_launch")
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.idx)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = [r.split(", ") for r in out.strip().splitlines() if r.count(",") >= 8]
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows), "power_w_max": max((float(r[3]) for r in rows
                                                         if r[3].replace(".", "").isdigit()),
                                                        default=None)}


def flush_l2(buf):
    buf.zero_()


# ------------------------------------------------------------------ our arm

class Runner:
    """Holds device buffers for one workload and runs its step."""

    def __init__(self, w, inp, fa):
        self.w, self.fa = w, fa
        d = torch.device("cuda")
        self.q, self.k, self.v = (inp[n].to(d) for n in ("q", "k", "v"))
        self.kv = None if inp["kv_len"] is None else inp["kv_len"].to(d)
        self.o = torch.empty_like(self.q)
        self.lse = torch.empty(self.q.shape[:3], dtype=torch.float32, device=d)
        self.backward = w.backward
        if self.backward:
            self.do = inp["do"].to(d)
            self.dq = torch.empty_like(self.q)
            self.dk, self.dv = torch.empty_like(self.k), torch.empty_like(self.k)
            self.ws = fa.workspace(w.B, w.H, w.N, w.d, d)

    def fwd(self):
        self.fa.fa_fwd_v(self.q, self.k, self.v, self.o, self.lse, self.w.scale, self.w.causal,
                         self.kv, self.w.window)

    def prep(self):
        self.fa.fa_bwd_prep(self.o, self.do, self.lse, self.ws)

    def main(self):
        self.fa.fa_bwd_dkdv_v(self.q, self.k, self.v, self.do, self.dk, self.dv, self.w.scale,
                              self.w.causal, self.kv, self.w.window, self.ws)

    def post(self):
        self.fa.fa_bwd_dq(self.dq, self.w.scale, self.ws)

    def phases(self):
        main, post = bwd_kernel_names(self.w.d)
        return [("fa_fwd_kernel", self.fwd)] + ([("bwd_pre_kernel", self.prep),
                                                 (main, self.main),
                                                 (post, self.post)]
                                                if self.backward else [])

    def step(self):
        for _, f in self.phases():
            f()


class DecodeRunner:
    """Split-KV decoding (fa_decode: the split kernel and the merge) for one
    decode workload."""

    def __init__(self, w, inp, fa):
        self.w, self.fa = w, fa
        d = torch.device("cuda")
        self.q, self.k, self.v = (inp[n].to(d) for n in ("q", "k", "v"))
        self.kv = None if inp["kv_len"] is None else inp["kv_len"].to(d)
        self.o = torch.empty_like(self.q)
        self.lse = torch.empty(self.q.shape[:3], dtype=torch.float32, device=d)
        self.splits = max(1, fa.fa_decode_splits(w.B, w.kv_heads, w.N))
        self.ws = torch.empty(fa.fa_decode_workspace_bytes(w.B, w.H, w.queries, w.d, self.splits),
                              dtype=torch.uint8, device=d)
        self.backward = False

    def run(self):
        self.fa.fa_decode(self.q, self.k, self.v, self.o, self.lse, self.w.scale, self.w.causal,
                          self.kv, self.w.window, self.splits, self.ws)

    def phases(self):
        return [("fa_decode", self.run)]

    def step(self):
        self.run()


class Fp8Runner:
    """The E4M3 forward (fa_fp8_quantize, then fa_fwd_fp8) for one workload."""

    def __init__(self, w, inp, fa):
        self.w, self.fa = w, fa
        d = torch.device("cuda")
        self.q, self.k, self.v = (inp[n].to(d) for n in ("q", "k", "v"))
        self.kv = None if inp["kv_len"] is None else inp["kv_len"].to(d)
        self.o = torch.empty_like(self.q)
        self.lse = torch.empty(self.q.shape[:3], dtype=torch.float32, device=d)
        self.buf = fa.fp8_buffers(w.B, w.H, w.kv_heads, w.N, w.d, d)
        self.backward = False

    def quant(self):
        self.fa.fa_fp8_quantize(self.q, self.k, self.v, self.buf)

    def fwd(self):
        self.fa.fa_fwd_fp8(self.buf, self.o, self.lse, self.w.scale, self.w.causal, self.kv,
                           self.w.window)

    def phases(self):
        return [("fp8_quantize", self.quant), ("fa_fwd_kernel", self.fwd)]

    def step(self):
        for _, f in self.phases():
            f()


def time_steps(runner, steps, flush=None, median=False):
    """Per-phase and per-step device times (ms) over `steps` timed steps.
    Per phase: the mean launch time, or with median=True the median."""
    phases = runner.phases()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(phases) + 1)]
          for _ in range(steps)]
    per_phase = {name: [] for name, _ in phases}
    step_ms = []
    for s in range(steps):
        if flush is not None:
            flush()
        ev[s][0].record()
        for i, (_, f) in enumerate(phases):
            f()
            ev[s][i + 1].record()
    torch.cuda.synchronize()
    for s in range(steps):
        for i, (name, _) in enumerate(phases):
            per_phase[name].append(ev[s][i].elapsed_time(ev[s][i + 1]))
        step_ms.append(ev[s][0].elapsed_time(ev[s][-1]))
    pick = statistics.median if median else (lambda v: sum(v) / len(v))
    return {k: pick(v) for k, v in per_phase.items()}, step_ms


def bytes_of(*ts):
    return sum(t.numel() * t.element_size() for t in ts if t is not None)


def run_ours(args, dist):
    from exact_attention_04_gb300 import build as fabuild
    from exact_attention_04_gb300 import fa

    fabuild.build()
    fa.load()
    torch.cuda.set_device(dist.local_rank)
    if args.sweep_only is not None:
        peaks, _ = load_peaks()
        return {"sweep": run_sweep(fa, peaks, only=args.sweep_only)}
    w = WORKLOADS[args.workload]
    if args.batch:
        w = dataclasses.replace(w, B=args.batch, name=f"{w.name}@B{args.batch}")
    if dist.rank:
        w = dataclasses.replace(w, seed=w.seed + 1000 * dist.rank)
    inp = make_inputs(w, with_grad_out=None if not args.fp8 else False)
    r = Fp8Runner(w, inp, fa) if args.fp8 else Runner(w, inp, fa)
    flops_fwd = w.fwd_flops()
    flops_bwd = w.bwd_flops() if r.backward else 0.0
    flops_step = flops_fwd + flops_bwd

    for _ in range(max(args.warmup, 3)):
        r.step()
    torch.cuda.synchronize()
    fa.fa_check()

    visible = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    clocks = ClockSampler(visible.split(",")[dist.local_rank] if visible else dist.local_rank)
    clocks.start()
    time.sleep(0.3)                      # let the sampler start
    for _ in range(max(args.warmup, 3)):
        r.step()                         # keep the GPU loaded while sampling begins
    dist.barrier()
    torch.cuda.synchronize()
    clocks.mark_start()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    per_phase, step_ms = time_steps(r, args.steps)
    end.record()
    torch.cuda.synchronize()
    dist.barrier()
    clocks.mark_end()
    clk = clocks.stop()
    fa.fa_check()
    total_ms = start.elapsed_time(end)
    total_ms = dist.max(total_ms)
    ms_per_step = total_ms / args.steps
    value = dist.world * flops_step / (ms_per_step * 1e-3) / 1e12

    # dominant kernel and its roofline
    peaks, peak_src = load_peaks()
    kernel = max(per_phase, key=per_phase.get)
    kflops = {"fa_fwd_kernel": flops_fwd, bwd_kernel_names(w.d)[0]: flops_bwd}
    if kernel in kflops:
        achieved = kflops[kernel] / (per_phase[kernel] * 1e-3) / 1e12
        peak = peaks["bf16_tflops"] * (2 if args.fp8 else 1)
        roof = {"kernel": kernel, "bound": "tensor", "achieved": round(achieved, 2),
                "peak": peak, "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4),
                "traffic": None if args.fp8 else committed_traffic(kernel, w.name),
                "peak_source": (f"{peak_src} bf16 dense, burst"
                                + (" x 2 (nominal E4M3 : BF16 dense ratio)" if args.fp8 else "")),
                "avg_launch_ms": round(per_phase[kernel], 4)}
    else:
        roof = {"kernel": kernel, "bound": "hbm", "achieved": None, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": None, "traffic": None}

    # end to end through the C ABI with pinned host buffers
    r2 = Fp8Runner(w, inp, fa) if args.fp8 else Runner(w, inp, fa)
    e2e = run_e2e([r, r2], w, fa, args.steps, flops_step, dist)
    del r2

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3" if args.fp8 else "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                   "causal": w.causal,
                   "pass": "fwd (E4M3)" if args.fp8 else ("fwd+bwd" if w.backward else "fwd"),
                   "parallelism": f"replica x{dist.world} (weak scaling, no collective)",
                   "l2": "inputs larger than L2, no flush"},
        "fwd_tflops": round(flops_fwd / (per_phase["fa_fwd_kernel"] * 1e-3) / 1e12, 2),
        "bwd_tflops": (round(flops_bwd / (sum(per_phase[k] for k in per_phase
                                               if k != "fa_fwd_kernel") * 1e-3) / 1e12, 2)
                       if r.backward else None),
        "kernel_ms": {k: round(v, 4) for k, v in per_phase.items()},
        "step_ms_median": round(statistics.median(step_ms), 4),
        "roofline": roof,
        "e2e": e2e,
        "gpu_launches": args.steps * len(r.phases()),
        "clocks": clk,
    }
    del r
    torch.cuda.empty_cache()
    if not args.no_sweep:
        result["sweep"] = run_sweep(fa, peaks)
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline and not args.fp8:
        result["cpu_baseline"] = cpu_baseline(w, inp)
    return result


def run_e2e(rs, w, fa, steps, flops_step, dist):
    """The same step end to end: every step copies its inputs from pinned host
    memory to the device and every output back (o, lse and, with the
    backward, dq, dk, dv), inside the timed region.  The copies run on their
    own streams and two device buffer sets alternate, so the inputs of step
    s+1 and the outputs of step s-1 move while step s computes.  The first
    step's upload and the last step's download overlap nothing and stay in
    the timed region; over `steps` steps they add about 1.3 ms / steps each
    step at the headline shape.

    rs: two runners of the workload (two device buffer sets)."""
    r0 = rs[0]
    hin = {n: getattr(r0, n).cpu().pin_memory() for n in (["q", "k", "v"] +
                                                          (["do"] if r0.backward else []))}
    outs = ["o", "lse"] + (["dq", "dk", "dv"] if r0.backward else [])
    hout = {n: torch.empty_like(getattr(r0, n), device="cpu").pin_memory() for n in outs}
    h2d = bytes_of(*hin.values())
    d2h = bytes_of(*hout.values())
    s_in, s_run, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()

    def run(n):
        ev = [[torch.cuda.Event() for _ in range(3)] for _ in range(n)]
        for k in range(n):
            r = rs[k % 2]
            with torch.cuda.stream(s_in):
                if k >= 2:
                    s_in.wait_event(ev[k - 2][1])       # step k-2 has consumed this set's inputs
                for name, t in hin.items():
                    getattr(r, name).copy_(t, non_blocking=True)
                ev[k][0].record(s_in)
            with torch.cuda.stream(s_run):
                s_run.wait_event(ev[k][0])
                if k >= 2:
                    s_run.wait_event(ev[k - 2][2])      # this set's outputs of step k-2 are copied out
                r.step()
                ev[k][1].record(s_run)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev[k][1])
                for name, t in hout.items():
                    t.copy_(getattr(r, name), non_blocking=True)
                ev[k][2].record(s_out)

    run(2)
    torch.cuda.synchronize()
    dist.barrier()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(s_in)
    run(steps)
    end.record(s_out)
    torch.cuda.synchronize()
    ms = dist.max(start.elapsed_time(end)) / steps
    fa.fa_check()
    return {"value": round(dist.world * flops_step / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 4),
            "steps": steps,
            "pipeline": "pinned host buffers; inputs of step s+1 and outputs of step s-1 copied on "
                        "their own streams while step s computes (two device buffer sets)"}


BLOCK_SPARSE = dict(B=2, H=16, N=8192, d=128, seed=12)
BLOCK_SPARSE_NAME = "blocksparse_b2_h16_n8192_d128_local_global_random"


class BlockSparseRunner:
    """Forward (fa_fwd_v) and backward (fa_bwd_v) of block-sparse attention:
    the local + global + random block pattern of block_sparse_mask.  balanced:
    pass the mask with its host copy (fa.BlockMask), so the launches plan a
    balanced tail on the host; else the device mask alone, whose tiles and key
    blocks the kernels sort by cost on the device (the cost-sorted deal)."""

    def __init__(self, fa, balanced=True):
        c = BLOCK_SPARSE
        self.w = random_case(c["B"], c["H"], c["N"], c["d"], seed=c["seed"], causal=False)
        inp = make_inputs(self.w)
        dev = torch.device("cuda")
        self.q, self.k, self.v, self.do = (inp[n].to(dev) for n in ("q", "k", "v", "do"))
        T = -(-c["N"] // 128)
        self.mask_np = block_sparse_mask(T, seed=c["seed"])
        self.mask = (fa.BlockMask(self.mask_np, dev) if balanced
                     else torch.from_numpy(self.mask_np).to(dev))
        self.o = torch.empty_like(self.q)
        self.lse = torch.empty(self.q.shape[:3], dtype=torch.float32, device=dev)
        self.dq, self.dk, self.dv = (torch.empty_like(self.q) for _ in range(3))
        self.ws = fa.workspace(c["B"], c["H"], c["N"], c["d"], dev)
        self.fa = fa

    def fwd(self):
        self.fa.fa_fwd_v(self.q, self.k, self.v, self.o, self.lse, self.w.scale,
                         block_mask=self.mask)

    def bwd(self):
        self.fa.fa_bwd_v(self.q, self.k, self.v, self.o, self.do, self.lse, self.dq, self.dk,
                         self.dv, self.w.scale, workspace=self.ws, block_mask=self.mask)

    def phases(self):
        return [("fwd", self.fwd), ("bwd", self.bwd)]

    def step(self):
        self.fwd()
        self.bwd()

    def computed_pairs(self):
        """(query, key) pairs the mask computes, per head (N a multiple of 128)."""
        return int(self.mask_np.sum()) * 128 * 128


def sweep_blocksparse(fa, peaks, flush_buf):
    timed = []
    for balanced in (True, False):
        r = BlockSparseRunner(fa, balanced)
        for _ in range(3):
            r.step()
        torch.cuda.synchronize()
        timed.append(time_steps(r, 20, flush=lambda: flush_l2(flush_buf), median=True)[0])
        fa.fa_check()
    per_phase, dev = timed
    c = BLOCK_SPARSE
    fwd_flops = 4.0 * c["B"] * c["H"] * c["d"] * r.computed_pairs()
    dense = 4.0 * c["B"] * c["H"] * c["d"] * c["N"] * c["N"]
    fwd_ms, bwd_ms = per_phase["fwd"], per_phase["bwd"]
    return {"workload": BLOCK_SPARSE_NAME,
            "N": c["N"], "d": c["d"], "causal": False,
            "block_density": round(float(r.mask_np.mean()), 4),
            "fwd_ms": round(fwd_ms, 4),
            "fwd_tflops": round(fwd_flops / (fwd_ms * 1e-3) / 1e12, 2),
            "fwd_frac_of_peak": round(fwd_flops / (fwd_ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
            "bwd_ms": round(bwd_ms, 4),
            "bwd_tflops": round(2.5 * fwd_flops / (bwd_ms * 1e-3) / 1e12, 2),
            "bwd_frac_of_peak": round(2.5 * fwd_flops / (bwd_ms * 1e-3) / 1e12
                                      / peaks["bf16_tflops"], 4),
            "dense_equivalent_tflops": round(dense / (fwd_ms * 1e-3) / 1e12, 2),
            "device_planned": {"fwd_ms": round(dev["fwd"], 4), "bwd_ms": round(dev["bwd"], 4),
                               "note": "the device mask alone (no host copy): the cost-sorted "
                                       "deal planned on the device"},
            "flops": "computed (query, key) pairs only: 4 d per pair forward, 2.5x backward",
            "timing": "median of 20 steps, L2 flushed before each"}


def visible_pairs(L, N, causal):
    """(query, key) pairs of one head that a key-padding length L leaves
    visible: every query sees keys j < L (and j <= i when causal)."""
    L = max(0, min(L, N))
    return L * (L + 1) // 2 + (N - L) * L if causal else N * L


def roofline_frac(flops, nbytes, ms, peaks):
    """Achieved FLOP/s over the roofline min(pi, AI * beta): pi the measured
    dense bf16 peak, beta the measured HBM bandwidth, AI = algorithmic FLOPs
    per algorithmic byte."""
    roof = min(peaks["bf16_tflops"] * 1e12, flops / nbytes * peaks["hbm_gbs"] * 1e9)
    return round(flops / (ms * 1e-3) / roof, 4)


def run_sweep(fa, peaks, only=None):
    """Every other workload, timed briefly: TFLOP/s, fraction of peak, GB/s of
    algorithmic traffic (inputs read + outputs written once).  only: keep the
    workloads whose name contains this string."""
    out = []
    flush_buf = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device="cuda")
    cache = {}
    for name, w in WORKLOADS.items():
        if only is not None and only not in name:
            continue
        if name == HEADLINE:
            inp = make_inputs(w, with_grad_out=False)
            out.append({"workload": name, "N": w.N, "d": w.d, "causal": w.causal,
                        "fp8": sweep_fp8(w, inp, fa, peaks, flush_buf)})
            del inp
            continue
        key = (w.B, w.H, w.kv_heads, w.queries, w.N, w.d, w.seed, w.qk_gain, w.kv_len_range,
               w.backward)
        if key not in cache:
            cache.clear()
            cache[key] = make_inputs(w)
        inp = cache[key]
        if w.nq is not None:
            out.append(sweep_decode(w, inp, fa, peaks, flush_buf))
            continue
        r = Runner(w, inp, fa)
        for _ in range(3):
            r.step()
        torch.cuda.synchronize()
        steps = 20
        per_phase, _ = time_steps(r, steps, flush=lambda: flush_l2(flush_buf), median=True)
        fa.fa_check()
        fwd_ms = per_phase["fa_fwd_kernel"]
        rowb = w.B * w.H * w.N               # query rows
        kvrowb = w.B * w.kv_heads * w.N      # key rows
        fwd_bytes = 4 * rowb * w.d + 4 * kvrowb * w.d + 4 * rowb     # Q, O; K, V; LSE
        entry = {"workload": name, "N": w.N, "d": w.d, "causal": w.causal,
                 "h_kv": w.kv_heads, "window": list(w.window) if w.window else None,
                 "fwd_ms": round(fwd_ms, 4),
                 "fwd_tflops": round(w.fwd_flops() / (fwd_ms * 1e-3) / 1e12, 2),
                 "fwd_frac_of_peak": round(w.fwd_flops() / (fwd_ms * 1e-3) / 1e12
                                           / peaks["bf16_tflops"], 4),
                 "fwd_gbs": round(fwd_bytes / (fwd_ms * 1e-3) / 1e9, 1),
                 "fwd_frac_of_roofline": roofline_frac(w.fwd_flops(), fwd_bytes, fwd_ms, peaks),
                 "timing": "median of 20 steps, L2 flushed before each"}
        if r.backward:
            bwd_ms = sum(v for k, v in per_phase.items() if k != "fa_fwd_kernel")
            bwd_bytes = 8 * rowb * w.d + 8 * kvrowb * w.d + 12 * rowb   # Q,O,dO,dQ; K,V,dK,dV
            entry.update({"bwd_ms": round(bwd_ms, 4),
                          "bwd_tflops": round(w.bwd_flops() / (bwd_ms * 1e-3) / 1e12, 2),
                          "bwd_frac_of_peak": round(w.bwd_flops() / (bwd_ms * 1e-3) / 1e12
                                                    / peaks["bf16_tflops"], 4),
                          "bwd_gbs": round(bwd_bytes / (bwd_ms * 1e-3) / 1e9, 1),
                          "bwd_frac_of_roofline": roofline_frac(w.bwd_flops(), bwd_bytes, bwd_ms,
                                                                peaks)})
        if w.backward and not r.backward:
            entry["bwd"] = "not built for this head dimension"
        if inp["kv_len"] is not None and w.window is None:
            # key padding: the headline convention counts every (query, key)
            # pair; this second figure counts only the pairs a query can see
            uf = 4.0 * w.H * w.d * sum(visible_pairs(int(L), w.N, w.causal)
                                       for L in inp["kv_len"].tolist())
            entry["useful_fwd_tflops"] = round(uf / (fwd_ms * 1e-3) / 1e12, 2)
            if r.backward:
                entry["useful_bwd_tflops"] = round(2.5 * uf / (bwd_ms * 1e-3) / 1e12, 2)
        del r
        torch.cuda.empty_cache()
        if w.d in (128, 256):
            entry["fp8"] = sweep_fp8(w, inp, fa, peaks, flush_buf)
        out.append(entry)
    if only is None or only in BLOCK_SPARSE_NAME:
        cache.clear()
        torch.cuda.empty_cache()
        out.append(sweep_blocksparse(fa, peaks, flush_buf))
    return out


def sweep_fp8(w, inp, fa, peaks, flush_buf):
    """The E4M3 forward of a workload: the quantiser (HBM-bound: reads Q, K, V
    in bf16, writes them in E4M3) and the FP8 attention kernel, whose FLOPs
    are the bf16 forward's, against an E4M3 peak of twice the measured bf16
    one (the nominal dense ratio, 4.5 / 2.25 PFLOP/s)."""
    r = Fp8Runner(w, inp, fa)
    for _ in range(3):
        r.step()
    torch.cuda.synchronize()
    per_phase, _ = time_steps(r, 20, flush=lambda: flush_l2(flush_buf), median=True)
    fa.fa_check()
    qb = w.B * w.H * w.N * w.d
    kb = w.B * w.kv_heads * w.N * w.d
    qbytes = 3 * qb + 6 * kb                  # bf16 read (2 B) + E4M3 write (1 B) per element
    fwd_ms, q_ms = per_phase["fa_fwd_kernel"], per_phase["fp8_quantize"]
    tfl = w.fwd_flops() / (fwd_ms * 1e-3) / 1e12
    peak = 2 * peaks["bf16_tflops"]
    del r
    torch.cuda.empty_cache()
    return {"fwd_ms": round(fwd_ms, 4), "fwd_tflops": round(tfl, 2),
            "fwd_frac_of_peak": round(tfl / peak, 4), "peak_tflops": round(peak, 1),
            "peak": "2 x measured bf16 burst (nominal E4M3 : BF16 dense ratio)",
            "quantize_ms": round(q_ms, 4),
            "quantize_gbs": round(qbytes / (q_ms * 1e-3) / 1e9, 1)}


def sweep_decode(w, inp, fa, peaks, flush_buf):
    """A decode workload: bound by reading K and V once, so GB/s against the
    measured HBM peak is the figure that matters.  Timed both ways the timing
    rule allows: back to back with K and V larger than L2 (the streamed cache
    leaves nothing for the next step to hit), and after an L2 flush, whose
    dirty lines are written back while the next step reads."""
    r = DecodeRunner(w, inp, fa)
    for _ in range(3):
        r.step()
    torch.cuda.synchronize()
    qrows = w.B * w.H * w.queries
    kv_bytes = 4 * w.B * w.kv_heads * w.N * w.d           # K and V, bf16, read once
    nbytes = kv_bytes + 4 * qrows * w.d + 4 * qrows       # + Q, O (bf16) and LSE
    per_phase, _ = time_steps(r, 20, flush=lambda: flush_l2(flush_buf), median=True)
    ms_flush = per_phase["fa_decode"]
    per_phase, _ = time_steps(r, 20, median=True)
    ms = per_phase["fa_decode"]
    fa.fa_check()
    l2 = getattr(torch.cuda.get_device_properties(0), "L2_cache_size", 129 * 10 ** 6)
    large = kv_bytes > 2 * l2
    if not large:                                         # only the flushed number is valid
        ms = ms_flush
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"workload": w.name, "N": w.N, "nq": w.queries, "d": w.d, "causal": w.causal,
            "h_kv": w.kv_heads, "splits": r.splits, "decode_ms": round(ms, 4),
            "decode_gbs": round(gbs, 1), "decode_frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4),
            "decode_tflops": round(w.fwd_flops() / (ms * 1e-3) / 1e12, 3),
            "decode_ms_after_l2_flush": round(ms_flush, 4),
            "decode_frac_of_hbm_after_l2_flush":
                round(nbytes / (ms_flush * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
            "bytes": nbytes,
            "l2": ("K and V larger than L2, back to back" if large else
                   "flushed between steps"),
            "timing": "median of 20 steps each way"}


# ------------------------------------------------------------------ the oracle as baseline

def oracle_sample(w, inp):
    """One head (b=0, h=0) of the workload, forward and (if the workload has
    one) backward, in the fp64 oracle on every host core."""
    import oracle
    f64 = {n: inp[n][0:1, 0:1].float().double().numpy() for n in ("q", "k", "v")}
    if w.backward:
        f64["do"] = inp["do"][0:1, 0:1].float().double().numpy()
    kv = None if inp["kv_len"] is None else [int(inp["kv_len"][0])]
    threads = oracle.default_threads()
    one = dataclasses.replace(w, B=1, H=1)
    flops = one.fwd_flops() + (one.bwd_flops() if w.backward else 0.0)

    def run():
        oracle.attention_fwd(f64["q"], f64["k"], f64["v"], w.scale, causal=w.causal, kv_len=kv,
                             threads=threads)
        if w.backward:
            oracle.attention_bwd(f64["q"], f64["k"], f64["v"], f64["do"], w.scale,
                                 causal=w.causal, kv_len=kv, threads=threads)
    desc = (f"head (b=0,h=0) of {w.name}: N={w.N}, d={w.d}, "
            f"{'forward+backward' if w.backward else 'forward'}, fp64")
    return run, flops, threads, desc


# the small configurations the fp64 oracle runs whole, every head
ORACLE_WHOLE = ("single_head_b1_h1_n256_d64", "bert_large_b16_h16_n512_d64_pad",
                "gpt2_small_b8_h12_n1024_d64_causal")


def oracle_whole(name):
    """Seconds and TFLOP/s of the fp64 oracle on a whole small workload
    (forward, and backward where the workload has one) on every host core."""
    import oracle
    w = WORKLOADS[name]
    inp = make_inputs(w)
    f64 = {n: inp[n].float().double().numpy() for n in ("q", "k", "v")}
    kv = None if inp["kv_len"] is None else [int(x) for x in inp["kv_len"].tolist()]
    threads = oracle.default_threads()
    t0 = time.perf_counter()
    oracle.attention_fwd(f64["q"], f64["k"], f64["v"], w.scale, causal=w.causal, kv_len=kv,
                         threads=threads)
    if w.backward:
        do = inp["do"].float().double().numpy()
        oracle.attention_bwd(f64["q"], f64["k"], f64["v"], do, w.scale, causal=w.causal,
                             kv_len=kv, threads=threads)
    sec = time.perf_counter() - t0
    flops = w.fwd_flops() + (w.bwd_flops() if w.backward else 0.0)
    return {"workload": name, "pass": "fwd+bwd" if w.backward else "fwd",
            "seconds": round(sec, 3), "tflops": round(flops / sec / 1e12, 6)}


def cpu_baseline(w, inp):
    """The oracle on one sampled head of the workload (its TFLOP/s is the
    line's value), the whole workload's time extrapolated from it (heads are
    independent and equal in work, so the time is linear in B*H), and the
    small configurations run whole."""
    run, flops, threads, desc = oracle_sample(w, inp)
    t0 = time.perf_counter()
    run()
    sec = time.perf_counter() - t0
    return {"value": round(flops / sec / 1e12, 6), "unit": "TFLOP/s", "cores": threads,
            "kind": "oracle", "sample": desc, "seconds": round(sec, 3),
            "extrapolated": {"seconds": round(sec * w.B * w.H, 3), "heads": w.B * w.H,
                             "note": "the sampled head's time x B*H heads"},
            "whole_small_configs": [oracle_whole(n) for n in ORACLE_WHOLE]}


def run_reference(args, dist):
    if dist.rank != 0:
        return None
    w = WORKLOADS[args.workload]
    inp = make_inputs(w)
    run, flops, threads, desc = oracle_sample(w, inp)
    for _ in range(args.warmup):
        run()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        run()
        times.append(time.perf_counter() - t0)
    sec = sum(times) / len(times)
    value = round(flops / sec / 1e12, 6)
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": dist.world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(sec * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                       "causal": w.causal, "pass": "fwd+bwd" if w.backward else "fwd",
                       "sample": desc},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads,
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    args = parse_args()
    dist = Dist()
    try:
        res = run_reference(args, dist) if args.impl == "reference" else run_ours(args, dist)
        if dist.rank == 0 and res is not None:
            print(json.dumps(res), flush=True)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
