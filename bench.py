#!/usr/bin/env python3
"""Benchmark of the ring-attention hot path on GB300.

A step is one pass of the whole path over one batch of synthetic input that is
already resident in HBM: the ring forward (fused fp32 LSE merge) followed by
the ring backward (D = rowsum(dO*O), the backward kernel, the dQ cast).  The
workload is the causal zigzag one: b=1, h=32, s=65536, d=128, 8 shards each
holding chunks r and 15-r of 16 chunks of 4096 tokens, bf16 q/k/v/dO drawn
from N(0, 1).

value: fwd+bwd attention TFLOP/s, causal-adjusted: forward 4*b*h*s*s*d/2 and
fwd+bwd 2.5x that; the algorithmic 3.5x figure and the forward alone are also
printed.  Inputs (2 GiB) are larger than L2, so no flush is needed between
steps.  One JSON line is printed by rank 0.

--impl reference times the fp64 CPU oracle on a bounded sample of the same
workload (the first tokens of one head: a causal prefix is an exact
sub-problem) on the host cores.
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
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention TFLOP/s (causal-adjusted) fwd and fwd+bwd; % of GB300 dense-BF16 peak"
B, H, S, D, N_SHARDS, LAYOUT = 1, 32, 65536, 128, 8, "zigzag"
SEED = 1003
WORKLOAD = "causal zigzag fwd+bwd: b1 h32 s65536 d128, 8 shards (chunks r and 15-r of 16 x 4096), bf16 N(0,1)"
FWD_FLOP = 4.0 * B * H * S * S * D / 2.0          # causal-adjusted forward
STEP_FLOP = 2.5 * FWD_FLOP                         # fwd+bwd, 2.5x convention
STEP_FLOP_ALG = 3.5 * FWD_FLOP                     # fwd + bwd (5 GEMMs vs 2)
BWD_FLOP = 2.5 * FWD_FLOP                          # backward alone: 10*d per unmasked pair
CPU_SAMPLE_TOKENS = 8192       # reference arm: one step of CPU work
CPU_BASELINE_TOKENS = 24576    # cpu_baseline: ~10-30 s of CPU work (about 12 s on 16 Arm cores)


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm": float(p["hbm_gbs"]), "bf16": float(p["bf16_tflops"]),
                "bf16_sustained": float(p["bf16_tflops_sustained"]), "source": "measured"}
    except Exception:
        return {"hbm": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "source": "fallback"}


def _kernel_source_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _profiled_traffic(kernel_file, src_files):
    """DRAM bytes per launch from the committed ncu summary, if the kernel is unchanged since."""
    path = os.path.join(ROOT, "profiles", kernel_file)
    try:
        text = open(path).read()
    except OSError:
        return None
    m = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    h = re.search(r"source_sha256_16:\s*([0-9a-f]+)", text)
    if not m or not h or h.group(1) != _kernel_source_hash(src_files):
        return None
    return float(m.group(1))


class ClockSampler:
    """nvidia-smi sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.path = os.path.join("/tmp", f"ra_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        try:
            os.remove(self.path)
        except OSError:
            pass
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(power) if power else None, "samples": len(sm), "reasons": sorted(reasons)}


def _cpu_threads():
    try:
        from threadpoolctl import threadpool_info

        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n and n[0]:
            return int(n[0])
    except Exception:
        pass
    return os.cpu_count()


def _oracle_sample(q, k, v, do):
    """The fp64 oracle (as it stands) on a causal prefix of one head; returns (seconds, flop)."""
    import oracle

    t0 = time.perf_counter()
    oracle.attention_fwd(q, k, v, D ** -0.5, True)
    oracle.attention_bwd(q, k, v, do, D ** -0.5, True)
    dt = time.perf_counter() - t0
    n = q.shape[2]
    return dt, 2.5 * 4.0 * n * n * D / 2.0


def max_over_ranks(x: float, dist, device) -> float:
    """The largest per-rank value (the job's time is its slowest rank's)."""
    if dist is None:
        return float(x)
    import torch

    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world: int, flop_per_rank_step: float, ms_per_step: float) -> float:
    """Whole-job throughput: every rank's work divided by the slowest rank's time."""
    return world * flop_per_rank_step / (ms_per_step * 1e-3) / 1e12


def _emit(obj):
    print(json.dumps(obj), flush=True)


# ----------------------------------------------------------------------------- reference arm
def reference_arm(args, rank, world):
    if rank != 0:
        return 0
    from workload import make_qkv

    x = make_qkv(1, 1, CPU_SAMPLE_TOKENS, D, SEED, with_do=True)
    q, k, v, do = (x[n] for n in ("q", "k", "v", "do"))
    for _ in range(args.warmup):
        _oracle_sample(q, k, v, do)
    total_t, total_f = 0.0, 0.0
    for _ in range(args.steps):
        dt, fl = _oracle_sample(q, k, v, do)
        total_t += dt
        total_f += fl
    val = total_f / total_t / 1e12
    sample = (f"fp64 numpy oracle, fwd+bwd of the causal prefix of {CPU_SAMPLE_TOKENS} tokens of one head "
              f"(an exact sub-problem of the workload), per step")
    _emit({"impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": args.gpus,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / args.steps,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": WORKLOAD, "sample_tokens": CPU_SAMPLE_TOKENS, "sample_heads": 1},
           "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": _cpu_threads(), "kind": "oracle",
                            "sample": sample},
           "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}})
    return 0


def _shrink(s, h):
    """A smaller case of the same workload (profiling captures); the JSON names it."""
    global S, H, FWD_FLOP, STEP_FLOP, STEP_FLOP_ALG, BWD_FLOP, WORKLOAD
    S, H = int(s), int(h)
    FWD_FLOP = 4.0 * B * H * S * S * D / 2.0
    STEP_FLOP, STEP_FLOP_ALG, BWD_FLOP = 2.5 * FWD_FLOP, 3.5 * FWD_FLOP, 2.5 * FWD_FLOP
    c = S // (2 * N_SHARDS)
    WORKLOAD = (f"causal zigzag fwd+bwd: b1 h{H} s{S} d128, 8 shards (chunks r and 15-r of 16 x {c}), "
                f"bf16 N(0,1) [reduced profiling case]")


# ----------------------------------------------------------------------------- our arm
def _varlen_leg(ra, torch, wid, peaks, dev, steps=5, warmup=3, heads=None):
    """fwd + bwd of a packed varlen workload, inputs resident in layout order,
    timed with CUDA events around `steps` steps on the current stream (heads:
    fewer heads, for profiling captures)."""
    import dataclasses

    from workload import WORKLOADS, cu_seqlens, make_workload_inputs

    w = WORKLOADS[wid]
    if heads:
        w = dataclasses.replace(w, h=int(heads))
    cu = torch.tensor(cu_seqlens(w.seq_lengths()), dtype=torch.int32)
    x = make_workload_inputs(w, device=str(dev))
    g = {n: ra.ring_attn_varlen_permute(t[0].contiguous(), cu, w.layout, w.n_shards, seq_dim=1) for n, t in x.items()}
    del x
    out = torch.empty_like(g["q"])
    lse = torch.empty((w.h, w.s), dtype=torch.float32, device=dev)
    dq, dk, dv = (torch.empty_like(g["q"]) for _ in range(3))
    # one workspace for both calls (the forward's copies are dead when the backward runs);
    # for zigzag it holds the original-order copies the library computes in
    ws_bytes = max(ra.ring_attn_varlen_workspace_size(op, w.s, w.h, w.d, w.layout, w.n_shards) for op in (0, 1))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    cuw = ra.CuSeqlens(cu, dev)  # host and device copies made once: the timed steps copy nothing

    def step():
        ra.ring_attn_varlen_fwd(g["q"], g["k"], g["v"], cuw, None, w.n_shards, w.causal, w.scale, out=out, lse=lse,
                                layout=w.layout, workspace=ws)
        ra.ring_attn_varlen_bwd(g["do"], g["q"], g["k"], g["v"], out, lse, cuw, None, w.n_shards, w.causal,
                                w.scale, dq=dq, dk=dk, dv=dv, workspace=ws, layout=w.layout)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    # per-kernel split, from a separate timed pass (the events sit between launches)
    ra.ring_attn_timing_enable(True)
    for _ in range(2):
        step()
    kt = {n: ra.ring_attn_timing_read(n) for n in ("fwd", "bwd_pre", "bwd_dkdv", "bwd_dq", "permute")}
    ra.ring_attn_timing_enable(False)
    st, info = ra.ring_attn_check_device_error()
    if st != 0:
        raise RuntimeError(f"device error {st} info {info:#x} in the varlen leg")
    tf = 2.5 * w.fwd_flops() / (ms * 1e-3) / 1e12
    steps_timed = 2  # the per-kernel pass above
    return {"workload": f"{w.name}: h{w.h} total {w.s} d{w.d}, {w.varlen_seqs} seqs, {w.n_shards} {w.layout} shards",
            "ms_per_step": ms, "tflops": tf, "frac_of_peak": tf / peaks["bf16_sustained"],
            "frac_of_burst": tf / peaks["bf16"],
            "kernel_ms": {n: t / max(c, 1) for n, (t, c) in kt.items() if n != "permute"},
            "permute_ms_per_step": kt["permute"][0] / steps_timed,
            "path": ("inputs copied from zigzag to original order inside the workspace, contiguous-layout kernels "
                     "writing their results in zigzag order" if w.layout == "zigzag" else "contiguous-layout kernels"),
            "flop_convention": "fwd = sum_k 4*h*L_k^2*d/2; fwd+bwd = 2.5 x fwd"}


def _batched_leg(ra, torch, wid, peaks, dev, steps=5, warmup=3):
    """One of the pages' batched workloads other than the headline one (the
    contiguous 16k forward, the stripe 128k forward+backward): inputs resident
    in layout order, `steps` steps timed with CUDA events on the current
    stream, then a separate pass split per kernel."""
    from workload import WORKLOADS, make_workload_inputs

    w = WORKLOADS[wid]
    x = make_workload_inputs(w, device=str(dev))
    g = {n: ra.ring_attn_permute(t, w.layout, w.n_shards) for n, t in x.items()}
    del x
    out = torch.empty_like(g["q"])
    lse = torch.empty((w.b, w.h, w.s), dtype=torch.float32, device=dev)
    if w.backward:
        dq, dk, dv = (torch.empty_like(g["q"]) for _ in range(3))
        ws = torch.empty(ra.ring_attn_workspace_size(1, w.b, w.h, w.s, w.d, w.n_shards), dtype=torch.uint8,
                         device=dev)

    def step():
        ra.ring_attn_fwd(g["q"], g["k"], g["v"], w.layout, w.n_shards, w.causal, w.scale, out=out, lse=lse)
        if w.backward:
            ra.ring_attn_bwd(g["do"], g["q"], g["k"], g["v"], out, lse, w.layout, w.n_shards, w.causal, w.scale,
                             dq=dq, dk=dk, dv=dv, workspace=ws)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    ra.ring_attn_timing_enable(True)
    for _ in range(2):
        step()
    names = ("fwd", "bwd_pre", "bwd_dkdv", "bwd_dq") if w.backward else ("fwd",)
    kt = {n: ra.ring_attn_timing_read(n) for n in names}
    ra.ring_attn_timing_enable(False)
    st, info = ra.ring_attn_check_device_error()
    if st != 0:
        raise RuntimeError(f"device error {st} info {info:#x} in the {w.name} leg")
    kms = {n: t / max(c, 1) for n, (t, c) in kt.items()}
    fwd_f = w.fwd_flops()
    fwd_tf = fwd_f / (kms["fwd"] * 1e-3) / 1e12
    res = {"workload": f"{w.name}: b{w.b} h{w.h} s{w.s} d{w.d}, {w.n_shards} {w.layout} shards, "
                       f"{'causal' if w.causal else 'non-causal'}",
           "fwd_tflops": fwd_tf, "fwd_frac_of_burst": fwd_tf / peaks["bf16"],
           "fwd_frac_of_sustained": fwd_tf / peaks["bf16_sustained"], "kernel_ms": kms, "ms_per_step": ms}
    if w.backward:
        tf = 2.5 * fwd_f / (ms * 1e-3) / 1e12
        res.update({"fwd_bwd_tflops": tf, "fwd_bwd_frac_of_burst": tf / peaks["bf16"],
                    "fwd_bwd_frac_of_sustained": tf / peaks["bf16_sustained"],
                    "fwd_bwd_tflops_3p5x": 3.5 * fwd_f / (ms * 1e-3) / 1e12,
                    "dkdv_tflops_performed": 2.0 * fwd_f / (kms["bwd_dkdv"] * 1e-3) / 1e12,
                    "dq_tflops_performed": 1.5 * fwd_f / (kms["bwd_dq"] * 1e-3) / 1e12})
    else:
        res["fwd_tflops_step"] = fwd_f / (ms * 1e-3) / 1e12
    res["flop_convention"] = "fwd = 4*b*h*s^2*d (/2 causal); fwd+bwd = 2.5 x fwd"
    return res


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-legs", action="store_true", help="skip the contiguous-16k and stripe-128k legs")
    ap.add_argument("--dkdv", choices=["pair", "one"], default=None,
                    help="dK / dV kernel at head_dim 128: CTA pairs or one CTA per key tile (default: the library's)")
    ap.add_argument("--seq", type=int, default=None, help="smaller sequence length (profiling cases only)")
    ap.add_argument("--heads", type=int, default=None, help="fewer heads (profiling cases only)")
    ap.add_argument("--varlen", type=int, choices=[5, 6], default=None,
                    help="run only the varlen leg of this workload and print its figures (profiling aid)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return reference_arm(args, rank, world)
    if args.seq or args.heads:
        _shrink(args.seq or S, args.heads or H)

    import torch

    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    if rank == 0:
        import __graft_entry__

        __graft_entry__.build()
    if dist is not None:
        dist.barrier()
    import ring_attn_gb300 as ra
    from workload import make_qkv

    ra.load()
    if args.dkdv:
        ra.ring_attn_set_knob(ra.RA_KNOB_DKDV_PAIR, 1 if args.dkdv == "pair" else 0)
    dev = torch.device("cuda", local)
    peaks = _peaks()
    if args.varlen:
        # profiling aid, not a bench line: one varlen workload (optionally fewer heads) alone
        res = _varlen_leg(ra, torch, args.varlen, peaks, dev, steps=args.steps, warmup=args.warmup, heads=args.heads)
        if rank == 0:
            _emit({"varlen_only": args.varlen, **res})
        return 0
    scale = D ** -0.5

    # inputs: seeded on the device, original order, then moved to layout order by the library
    x = make_qkv(B, H, S, D, SEED + 1000 * rank, with_do=True, device=str(dev))
    ra.ring_attn_timing_enable(True)
    g = {n: ra.ring_attn_permute(t, LAYOUT, N_SHARDS) for n, t in x.items()}
    torch.cuda.synchronize()
    ra.ring_attn_timing_read("permute")
    q, k, v, do = g["q"], g["k"], g["v"], g["do"]
    out = torch.empty_like(q)
    lse = torch.empty((B, H, S), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(ra.ring_attn_workspace_size(1, B, H, S, D, N_SHARDS), dtype=torch.uint8, device=dev)

    def step():
        ra.ring_attn_fwd(q, k, v, LAYOUT, N_SHARDS, True, scale, out=out, lse=lse)
        ra.ring_attn_bwd(do, q, k, v, out, lse, LAYOUT, N_SHARDS, True, scale, dq=dq, dk=dk, dv=dv, workspace=ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st, info = ra.ring_attn_check_device_error()
    if st != 0:
        raise RuntimeError(f"device error {st} info {info:#x} during warm-up")
    for kname in ra.KERNELS:
        ra.ring_attn_timing_read(kname)

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    clk = clocks.stop()
    ms = e0.elapsed_time(e1) / args.steps
    kt = {kname: ra.ring_attn_timing_read(kname) for kname in ra.KERNELS}
    launches = sum(n for _, n in kt.values())
    st, info = ra.ring_attn_check_device_error()
    if st != 0:
        raise RuntimeError(f"device error {st} info {info:#x} in the timed region")
    ms = max_over_ranks(ms, dist, dev)

    def avg(name):
        return kt[name][0] / max(kt[name][1], 1)

    fwd_ms, dkdv_ms, dq_ms, pre_ms = avg("fwd"), avg("bwd_dkdv"), avg("bwd_dq"), avg("bwd_pre")
    bwd_ms = dkdv_ms + dq_ms + pre_ms
    value = job_tflops(world, STEP_FLOP, ms)
    bwd_tflops = BWD_FLOP / (bwd_ms * 1e-3) / 1e12
    fwd_tflops = FWD_FLOP / (fwd_ms * 1e-3) / 1e12
    peak_sus = peaks["bf16_sustained"]
    # FLOP each kernel performs: forward 2 GEMMs, dK/dV 4 GEMMs, dQ 3 GEMMs (S and dP recomputed)
    bwd_src = ["ring_attn_gb300/csrc/ra_bwd.cu", "ring_attn_gb300/csrc/ra_bwd_common.cuh"]
    kernels = {
        "ring_fwd_kernel<128>": (fwd_ms, FWD_FLOP, ["ring_attn_gb300/csrc/ra_fwd.cu"], "ring_fwd_kernel_zigzag_h32_s64k.md"),
        "ring_dkdv_kernel<128>": (dkdv_ms, 2.0 * FWD_FLOP, bwd_src, "ring_dkdv_kernel_zigzag_h32_s64k.md"),
        "ring_dq_kernel<128>": (dq_ms, 1.5 * FWD_FLOP, bwd_src, "ring_dq_kernel_zigzag_h32_s64k.md"),
    }
    common = ["ring_attn_gb300/csrc/ra_device.cuh", "ring_attn_gb300/csrc/ra_internal.h",
              "ring_attn_gb300/csrc/ra_tiles.cuh"]
    dom = max(kernels, key=lambda k: kernels[k][0])
    d_ms, d_flop, d_src, d_prof = kernels[dom]
    d_tflops = d_flop / (d_ms * 1e-3) / 1e12
    roofline = {"kernel": dom, "bound": "tensor", "achieved": d_tflops, "peak": peak_sus, "unit": "TFLOP/s",
                "frac": d_tflops / peak_sus, "traffic": _profiled_traffic(d_prof, d_src + common),
                "frac_of_burst": d_tflops / peaks["bf16"],
                "algorithmic_flop_per_launch": d_flop, "peak_kind": f"bf16 sustained ({peaks['source']})",
                "launch_ms": d_ms}
    result = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1), cast to bf16)",
        "config": {"workload": WORKLOAD, "b": B, "h": H, "s": S, "d": D, "layout": LAYOUT, "n_shards": N_SHARDS,
                   "causal": True, "flop_convention": "fwd = 4*b*h*s^2*d/2; fwd+bwd = 2.5 x fwd",
                   "l2": "no flush: inputs larger than L2 (q, k, v, dO 512 MiB each)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "fwd": {"tflops": fwd_tflops, "ms": fwd_ms, "frac_of_peak": fwd_tflops / peak_sus,
                "frac_of_burst": fwd_tflops / peaks["bf16"],
                "traffic": _profiled_traffic("ring_fwd_kernel_zigzag_h32_s64k.md",
                                             ["ring_attn_gb300/csrc/ra_fwd.cu"] + common)},
        "bwd": {"tflops": bwd_tflops, "ms": bwd_ms, "frac_of_peak": bwd_tflops / peak_sus,
                "flop_credited": "2.5 x forward (the 5 backward GEMMs; the 2 recomputed in the dQ pass are not)",
                "dkdv_ms": dkdv_ms, "dkdv_tflops_performed": 2.0 * FWD_FLOP / (dkdv_ms * 1e-3) / 1e12,
                "dq_ms": dq_ms, "dq_tflops_performed": 1.5 * FWD_FLOP / (dq_ms * 1e-3) / 1e12, "pre_ms": pre_ms},
        "fwd_bwd_frac_of_peak": value / world / peak_sus,
        "fwd_bwd_frac_of_burst": value / world / peaks["bf16"],
        "fwd_bwd_tflops_3p5x": job_tflops(world, STEP_FLOP_ALG, ms),
        "roofline": roofline, "gpu_launches": launches, "clocks": clk,
        "peaks": peaks,
    }

    # ---- lse_merge standalone on the workload's full shape (HBM-bound)
    oacc = torch.zeros((B, H, S, D), dtype=torch.float32, device=dev)
    lacc = torch.full((B, H, S), -float("inf"), dtype=torch.float32, device=dev)
    ra.lse_merge(oacc, lacc, out, lse)
    torch.cuda.synchronize()
    ra.ring_attn_timing_read("lse_merge")
    for _ in range(5):
        ra.lse_merge(oacc, lacc, out, lse)
    m_ms, m_n = ra.ring_attn_timing_read("lse_merge")
    rows = B * H * S
    m_bytes = rows * (4 * D + 4 + 2 * D + 4 + 4 * D + 4)
    m_gbs = m_bytes / (m_ms / m_n * 1e-3) / 1e9
    result["lse_merge"] = {"gbs": m_gbs, "frac_of_hbm": m_gbs / peaks["hbm"], "bytes_per_call": m_bytes,
                           "ms": m_ms / m_n, "rows": rows}
    del oacc, lacc
    # ---- permute
    for n, t in x.items():
        ra.ring_attn_permute(t, LAYOUT, N_SHARDS, out=g[n])
    p_ms, p_n = ra.ring_attn_timing_read("permute")
    p_bytes = 2 * q.numel() * 2
    result["permute"] = {"gbs": p_bytes / (p_ms / p_n * 1e-3) / 1e9, "ms": p_ms / p_n,
                         "frac_of_hbm": p_bytes / (p_ms / p_n * 1e-3) / 1e9 / peaks["hbm"]}
    ra.ring_attn_timing_enable(False)

    # ---- varlen workloads (64 packed sequences, one cu_seqlens), contiguous and zigzag shards
    if not (args.seq or args.heads):
        result["varlen"] = {k: _varlen_leg(ra, torch, k, peaks, dev) for k in (5, 6)}

    # ---- e2e: host buffers in original order -> device -> permute -> fwd -> bwd -> unpermute -> host.
    # Every step uploads its four inputs from pinned host memory and reads all
    # five results back.  Uploads run on one copy stream and downloads on
    # another, into double-buffered device staging, so the copies of one step
    # overlap the compute of its neighbours (and dO's upload the forward).
    if not args.no_e2e:
        hin = {n: t.cpu().pin_memory() for n, t in x.items()}
        names_out = ("out", "dq", "dk", "dv")
        hout = {n: torch.empty_like(hin["q"]).pin_memory() for n in names_out}
        hlse = torch.empty((B, H, S), dtype=torch.float32).pin_memory()
        dbuf = [{n: torch.empty_like(x["q"]) for n in x} for _ in range(2)]
        rbuf = [{n: torch.empty_like(x["q"]) for n in names_out} for _ in range(2)]
        lbuf = [torch.empty_like(lse) for _ in range(2)]
        comp = torch.cuda.current_stream()
        up, down = torch.cuda.Stream(), torch.cuda.Stream()
        ev_in = [{n: torch.cuda.Event() for n in x} for _ in range(2)]   # input n of buffer j uploaded
        ev_used = [torch.cuda.Event() for _ in range(2)]                 # buffer j's inputs permuted
        ev_out = [torch.cuda.Event() for _ in range(2)]                  # buffer j's results unpermuted
        ev_read = [torch.cuda.Event() for _ in range(2)]                 # buffer j's results downloaded

        def e2e_step(i):
            j = i % 2
            up.wait_event(ev_used[j])
            with torch.cuda.stream(up):
                for n in ("q", "k", "v", "do"):
                    dbuf[j][n].copy_(hin[n], non_blocking=True)
                    ev_in[j][n].record(up)
            for n in ("q", "k", "v", "do"):
                comp.wait_event(ev_in[j][n])
                ra.ring_attn_permute(dbuf[j][n], LAYOUT, N_SHARDS, out=g[n])
            ev_used[j].record(comp)
            step()
            comp.wait_event(ev_read[j])
            for n, src in zip(names_out, (out, dq, dk, dv)):
                ra.ring_attn_unpermute(src, LAYOUT, N_SHARDS, out=rbuf[j][n])
            ra.ring_attn_unpermute(lse, LAYOUT, N_SHARDS, out=lbuf[j])
            ev_out[j].record(comp)
            down.wait_event(ev_out[j])
            with torch.cuda.stream(down):
                for n in names_out:
                    hout[n].copy_(rbuf[j][n], non_blocking=True)
                hlse.copy_(lbuf[j], non_blocking=True)
                ev_read[j].record(down)

        for i in range(2):
            e2e_step(i)
        comp.wait_stream(down)
        torch.cuda.synchronize()
        k_e2e = max(3, min(args.steps, 10))
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record()
        for i in range(k_e2e):
            e2e_step(i)
        comp.wait_stream(down)
        comp.wait_stream(up)
        a1.record()
        torch.cuda.synchronize()
        e_ms = a0.elapsed_time(a1) / k_e2e
        e_ms = max_over_ranks(e_ms, dist, dev)
        h2d = sum(t.numel() * t.element_size() for t in hin.values())
        d2h = sum(t.numel() * t.element_size() for t in hout.values()) + hlse.numel() * 4
        result["e2e"] = {"value": job_tflops(world, STEP_FLOP, e_ms), "unit": "TFLOP/s",
                         "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e_ms,
                         "steps": k_e2e,
                         "path": "pinned host -> C-ABI permute, fwd, bwd, unpermute -> pinned host; uploads and "
                                 "downloads on two copy streams, double-buffered, overlapping the compute"}

    # ---- CPU oracle baseline (rank 0, one GPU)
    if rank == 0 and world == 1 and not args.no_cpu:
        n = min(CPU_BASELINE_TOKENS, S)
        sample = {nm: t[:, :1, :n].cpu() for nm, t in x.items()}
        dt, fl = _oracle_sample(sample["q"], sample["k"], sample["v"], sample["do"])
        result["cpu_baseline"] = {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": _cpu_threads(),
                                  "kind": "oracle", "seconds": dt,
                                  "sample": f"fp64 numpy oracle fwd+bwd of the causal prefix of {n} tokens of "
                                            f"head 0 (exact sub-problem), same 2.5x flop convention"}
    # ---- the pages' other batched workloads: contiguous 16k forward, stripe 128k fwd+bwd
    if not (args.seq or args.heads or args.no_legs):
        del x, g, q, k, v, do, out, lse, dq, dk, dv, ws
        if not args.no_e2e:
            del hin, hout, hlse, dbuf, rbuf, lbuf
        torch.cuda.empty_cache()
        result["config2"] = _batched_leg(ra, torch, 2, peaks, dev)
        result["config4"] = _batched_leg(ra, torch, 4, peaks, dev)
    if rank == 0:
        _emit(result)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
