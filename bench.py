#!/usr/bin/env python
"""Throughput of one forward+backward step of bounded-decay chunked linear
attention through libbdla.so (C ABI), on synthetic inputs shaped like the
64K context stage (packed, 8 documents, H=32, dk=dv=128, bf16).

Prints ONE JSON line (rank 0).  `--impl reference` times the fp64 CPU oracle
on a bounded sample of the same workload instead (the only reference there
is: the pages ship no code).

Launch for N GPUs: python -m torch.distributed.run --nproc-per-node N
--master-addr 127.0.0.1 bench.py --gpus N.  Every rank runs its own replica
of the workload (units are independent; no data-path collective): weak
scaling, value = tokens of all ranks / max time over ranks.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "tokens/s fwd+bwd (T=64K,H=32,d=128 bf16); % of HBM/tensor-pipe roofline"
UNIT = "tokens/s"
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    # about 0.9 s of timed steps on the default workload, so that the clock
    # sampler (every 50 ms) sees the timed region many times over
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="varlen64k")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-ablation", action="store_true",
                    help="skip the 1M-token bounded-vs-ablation comparison")
    ap.add_argument("--variant", choices=["vec", "delta"], default=None,
                    help="run the workload's shape with one decay per key channel or as the gated delta rule")
    ap.add_argument("--ckpt-stride", type=int, default=None,
                    help="fp32 state checkpoints every N tokens (overrides the workload's own)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target CPU time of the oracle sample")
    return ap.parse_args()


def dist_env():
    from chunked_linear_attention_bounded_gb300.replicas import rank_env
    e = rank_env()
    return e.rank, e.world, e.local


def config_of(w, world):
    """The workload description both arms print."""
    tokens = w.B * w.T
    return {"workload": w.name, "tokens": tokens, "docs": w.n_docs if w.n_docs else w.B,
            "H": w.H, "dk": w.dk, "dv": w.dv,
            "decay": "bounded b*sigmoid(a), b=%g" % w.b if w.mode == 0 else "-softplus(a)",
            "l2": "inputs larger than L2 (q,k,v,dO bf16: %.2f GB)" % (4 * tokens * w.H * w.dk * 2 / 1e9),
            "parallelism": f"replicas x{world}"}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------- algorithmic bytes
def algorithmic_bytes(w, n_seq):
    """Bytes the method must move at minimum (fwd, bwd, per kernel).  With
    fp32 state checkpoints every `ckpt_stride` tokens (a config that asks for
    them), the checkpoints are outputs: the forward writes the 128-token block
    starts, the expansion kernel ("states") the ones inside each block, and
    the backward reads one per block."""
    th = w.B * w.T * w.H
    units = n_seq * w.H
    st = w.dk * w.dv * 4
    fwd = th * (2 * w.dk * 2 + 2 * w.dv + 4 + 2 * w.dv) + units * st * (2 if w.h0_std else 1)
    bwd = th * (2 * w.dk * 2 + 2 * w.dv * 2 + 4 + 4 * w.dk * 2 + 4 * w.dv + 4) + \
        (units * st if w.h0_std else 0)
    decay = th * 8
    out = {"fwd": fwd, "bwd": bwd, "decay": decay}
    if w.ckpt_stride and w.ckpt_stride < 128:
        per_block = 128 // w.ckpt_stride
        blocks = w.B * w.T // 128 * w.H
        out["fwd"] = fwd + blocks * st
        # k, v (bf16) and the tile cumsums read; the inner checkpoints written
        out["states"] = th * (2 * w.dk + 2 * w.dv + 4) + blocks * (per_block - 1) * st
        out["bwd"] = bwd + blocks * st
    return out


# ---------------------------------------------------------------- DRAM traffic
# dram__bytes_read.sum + dram__bytes_write.sum per launch from one ncu capture
# of the bench's own command (single-pass metrics, full-size workload), with a
# digest of the kernel source the capture ran.  Reported only while that
# source is unchanged; null otherwise.
NCU_TRAFFIC = {
    ("fwd", "varlen64k"): (1645925120 + 1054943488, "5f12712a3a3732fe"),
    ("bwd", "varlen64k"): (2716671744 + 3184528128, "9bad83a0b25edaef"),
    ("decode", "decode"): (543214336 + 478266112, "50dec6dabf6b63df"),
}
KERNEL_SOURCES = {
    "fwd": ("bdla_fwd_sm100.cu", "bdla_sm100.cuh", "bdla_common.cuh"),
    "bwd": ("bdla_bwd_sm100.cu", "bdla_sm100.cuh", "bdla_common.cuh"),
    "decode": ("bdla_decode.cu", "bdla_common.cuh"),
}


def kernel_digest(kernel: str) -> str:
    import hashlib
    csrc = os.path.join(ROOT, "chunked_linear_attention_bounded_gb300", "csrc")
    m = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, f), "rb") as fh:
            m.update(fh.read())
    return m.hexdigest()[:16]


def measured_traffic(kernel: str, workload: str):
    entry = NCU_TRAFFIC.get((kernel, workload))
    if entry is None or kernel_digest(kernel) != entry[1]:
        return None
    return entry[0]


def traffic_source(kernel: str, workload: str):
    """Where `traffic` comes from: a stored ncu capture, valid only for the
    kernel source it was taken on."""
    entry = NCU_TRAFFIC.get((kernel, workload))
    if entry is None:
        return "no ncu capture for this kernel and workload"
    if kernel_digest(kernel) != entry[1]:
        return f"ncu capture of source digest {entry[1]}; the source has changed since (digest {kernel_digest(kernel)})"
    return (f"ncu capture (dram__bytes_read.sum + dram__bytes_write.sum, one launch) of kernel source digest "
            f"{entry[1]}, not measured in this run")


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.gpu)], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- CPU oracle sample
def size_oracle_sample(inp, w, target_s: float):
    """Chooses a bounded sample of the workload for the fp64 oracle (as it
    stands): a prefix of the packed token stream (its documents cut at the
    prefix end) on a subset of the heads, grown until one fwd+bwd pass takes
    about `target_s` seconds.  Returns (run, ntok, nh, seconds of the last
    sizing pass); run() executes one fwd+bwd pass and returns its seconds."""
    import numpy as np

    import oracle
    threads = oracle.threads_used()
    cu_full = (inp["cu_seqlens"].numpy().astype(np.int64) if inp.get("cu_seqlens") is not None
               else np.arange(w.B + 1, dtype=np.int64) * w.T)
    total = int(cu_full[-1])

    def prepare(ntok, nh):
        cu = np.concatenate([cu_full[cu_full < ntok], [ntok]])
        sl = lambda t: t.reshape(-1, *t.shape[2:])[:ntok, :nh].double().numpy()
        q, k, v, dO = (sl(inp[x]) for x in ("q", "k", "v", "dO"))
        a = inp["a"].reshape(-1, w.H)[:ntok, :nh].double().numpy()
        h0 = None
        if inp.get("h0") is not None:
            h0 = inp["h0"][:len(cu) - 1, :nh].double().numpy()

        def run():
            t0 = time.perf_counter()
            oracle.fwd(q, k, v, a, w.b, w.mode, h0=h0, cu_seqlens=cu)
            oracle.bwd(q, k, v, a, dO, w.b, w.mode, h0=h0, cu_seqlens=cu)
            return time.perf_counter() - t0
        return run

    ntok, nh = min(total, 1024), min(w.H, threads)
    dt = prepare(ntok, nh)()
    grow = target_s / max(dt, 1e-4)
    # heads first (whole multiples of the thread count), then the prefix
    nh2 = min(w.H, max(nh, int(nh * grow) // threads * threads))
    grow *= nh / nh2
    ntok, nh = int(min(total, max(ntok, ntok * grow))), nh2
    run = prepare(ntok, nh)
    dt = run()
    if dt < 0.6 * target_s and ntok < total:      # the small first pass overstates the rate
        ntok = int(min(total, ntok * target_s / max(dt, 1e-4)))
        run = prepare(ntok, nh)
        dt = run()
    return run, ntok, nh, dt


def sample_desc(w, ntok, nh, dt):
    return (f"first {ntok} tokens of the packed stream x {nh} of {w.H} heads, fwd+bwd, "
            f"{dt:.1f} s per pass; tokens/s counts a token as all {w.H} heads")


def oracle_sample(inp, w, target_s: float):
    """One timed oracle pass on a sample sized for `target_s` seconds.
    Returns (tokens/s equivalent, cores, description)."""
    import oracle
    _, ntok, nh, dt = size_oracle_sample(inp, w, target_s)
    return ntok * nh / w.H / dt, oracle.threads_used(), sample_desc(w, ntok, nh, dt)


# ---------------------------------------------------------------- arms
def reference_arm(args, w, inp):
    """The reference arm: the fp64 oracle on the host cores, each step one
    fwd+bwd pass over the same bounded sample of the workload."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    per_step = max(0.5, min(args.cpu_seconds, 120.0 / max(1, args.steps + args.warmup)))
    run, ntok, nh, dt = size_oracle_sample(inp, w, per_step)
    for _ in range(args.warmup):
        run()
    times = [run() for _ in range(args.steps)]
    wall = sum(times)
    value = ntok * nh / w.H * args.steps / wall
    desc = sample_desc(w, ntok, nh, wall / args.steps)
    out = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": 1000.0 * wall / args.steps,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic", "impl": "reference",
           "config": config_of(w, world),
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.threads_used(),
                            "kind": "oracle", "sample": desc},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
           "gpu_launches": 0}
    print(json.dumps(out), flush=True)


def ours_arm(args, w, inp):
    import torch
    import torch.distributed as dist

    import chunked_linear_attention_bounded_gb300 as bdla
    from chunked_linear_attention_bounded_gb300 import bdla as B
    from chunked_linear_attention_bounded_gb300 import replicas

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    bdla.lib()
    g = {k: (v.to(dev) if v is not None else None) for k, v in inp.items()}
    n_seq = (g["cu_seqlens"].numel() - 1) if g["cu_seqlens"] is not None else w.B
    ws_f = B.Workspace(B.workspace_bytes(B.OP_FWD, tuple(g["q"].shape), w.dv, n_seq if g["cu_seqlens"] is not None else 0, w.mode), dev)
    # the forward hands the backward bf16 states every 128 tokens, unless the
    # config asks for fp32 state checkpoints at a finer stride: then those are
    # written (block starts by the forward, the rest by the expansion kernel)
    # and the backward reads them
    stride = w.ckpt_stride if w.ckpt_stride else 128
    ck_dtype = torch.float32 if w.ckpt_stride else torch.bfloat16
    ws_b = B.Workspace(B.workspace_bytes(B.OP_BWD, tuple(g["q"].shape), w.dv, n_seq if g["cu_seqlens"] is not None else 0, w.mode, ckpt_stride=stride), dev)
    o = torch.empty(g["v"].shape, dtype=torch.bfloat16, device=dev)
    ck = torch.empty((w.H, B.n_slots(w.B * w.T, n_seq, stride), w.dk, w.dv), dtype=ck_dtype, device=dev)
    hT = torch.empty((n_seq, w.H, w.dk, w.dv), dtype=torch.float32, device=dev)
    outs = (torch.empty(g["q"].shape, dtype=torch.float32, device=dev),
            torch.empty(g["k"].shape, dtype=torch.float32, device=dev),
            torch.empty(g["v"].shape, dtype=torch.float32, device=dev),
            torch.empty(g["a"].shape, dtype=torch.float32, device=dev))
    stream = torch.cuda.current_stream()

    def step(src):
        bdla.fwd(src["q"], src["k"], src["v"], src["a"], w.b, h0=src["h0"],
                 cu_seqlens=src["cu_seqlens"], mode=w.mode, ws=ws_f, out=o, hT_out=hT,
                 ckpt_stride=stride, ckpt_dtype=ck_dtype, ckpt_out=ck)
        bdla.bwd(src["q"], src["k"], src["v"], src["a"], src["dO"], w.b, h0=src["h0"],
                 cu_seqlens=src["cu_seqlens"], ckpt=ck, ckpt_stride=stride, mode=w.mode, ws=ws_b,
                 outs=outs)

    kernels = {"decay": B.KERNEL_DECAY, "fwd": B.KERNEL_FWD, "bwd": B.KERNEL_BWD,
               "states": B.KERNEL_STATES, "seg": B.KERNEL_SEG}
    seg = B.segments_engaged(tuple(g["q"].shape), w.dv, n_seq if g["cu_seqlens"] is not None else 0)
    # fwd: decay + fwd;  bwd: decay + bwd;  packed documents without segments:
    # the document order in each;  segments: summary + scan in each;  dv = 256:
    # the backward adds the second slice's partial sums
    ordered = g["cu_seqlens"] is not None and not seg and 1 < n_seq <= 4096
    # fp32 checkpoints inside the 128-token blocks: one expansion launch
    launches_per_step = 4 + (2 if ordered else 0) + (4 if seg else 0) + (1 if w.dv > 128 else 0) + \
        (1 if w.ckpt_stride and w.ckpt_stride < 128 else 0)

    def barrier():
        replicas.barrier(world)

    for _ in range(max(3, args.warmup)):
        step(g)
    torch.cuda.synchronize()
    for code in (ws_f.read_device_status(), ws_b.read_device_status()):
        if code:
            raise RuntimeError(f"device status {code} after warm-up")

    K = args.steps
    kev = {n: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)] for n in kernels}
    for pairs in kev.values():      # torch creates the CUDA event on first record
        for a_, b_ in pairs:
            a_.record(stream)
            b_.record(stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        e0.record(stream)
        for i in range(K):
            for n, kid in kernels.items():
                B.set_kernel_events(kid, *kev[n][i])
            step(g)
        e1.record(stream)
        torch.cuda.synchronize()
    barrier()
    for kid in kernels.values():
        B.set_kernel_events(kid, None, None)
    ms = replicas.max_over_ranks(e0.elapsed_time(e1) / K, world, dev)
    kernel_ms = {n: sum(a.elapsed_time(b) for a, b in kev[n]) / K for n in kernels}

    # end to end through the public API with host buffers: every step copies
    # its inputs from pinned host memory and its outputs (o, hT, dq, dk, dv, da)
    # back.  Copies run on their own streams with two sets of device buffers,
    # so one step's transfers overlap its neighbours' compute.
    host_in = {k: (v.pin_memory() if v is not None else None) for k, v in inp.items()}
    out_set = lambda: (torch.empty_like(o), torch.empty_like(hT), *(torch.empty_like(t) for t in outs))
    dev_outs = [(o, hT, *outs), out_set()]
    host_out = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in dev_outs[0]]
                for _ in range(2)]
    dev_in = [{k: (torch.empty_like(v, device=dev) if v is not None else None) for k, v in inp.items()}
              for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in host_in.values() if v is not None)
    d2h = sum(t.numel() * t.element_size() for t in host_out[0])
    # copies spread over several streams per direction (one large tensor each)
    n_in, n_out = 2, 3
    s_in = [torch.cuda.Stream(dev) for _ in range(n_in)]
    s_out = [torch.cuda.Stream(dev) for _ in range(n_out)]
    ev = lambda: torch.cuda.Event()
    h2d_done = [[ev() for _ in range(n_in)] for _ in range(2)]
    d2h_done = [[ev() for _ in range(n_out)] for _ in range(2)]
    comp_done = [ev(), ev()]
    # inputs split over the copy-in streams by size (largest first, to the lighter stream)
    in_groups, loads = [[] for _ in range(n_in)], [0] * n_in
    for k_, v_ in sorted(((k_, v_) for k_, v_ in host_in.items() if v_ is not None),
                         key=lambda kv: -kv[1].numel() * kv[1].element_size()):
        gi = loads.index(min(loads))
        in_groups[gi].append(k_)
        loads[gi] += v_.numel() * v_.element_size()

    def step_into(src, dst):
        do, dhT_, dq_, dk_, dv_, da_ = dst
        bdla.fwd(src["q"], src["k"], src["v"], src["a"], w.b, h0=src["h0"],
                 cu_seqlens=src["cu_seqlens"], mode=w.mode, ws=ws_f, out=do, hT_out=dhT_,
                 ckpt_stride=stride, ckpt_dtype=ck_dtype, ckpt_out=ck)
        bdla.bwd(src["q"], src["k"], src["v"], src["a"], src["dO"], w.b, h0=src["h0"],
                 cu_seqlens=src["cu_seqlens"], ckpt=ck, ckpt_stride=stride, mode=w.mode, ws=ws_b,
                 outs=(dq_, dk_, dv_, da_))

    def e2e_run(n):
        for i in range(n):
            b = i & 1
            for si, st_ in enumerate(s_in):
                with torch.cuda.stream(st_):
                    if i >= 2:
                        st_.wait_event(comp_done[b])      # step i-2 is done with these inputs
                    for k_ in in_groups[si]:
                        dev_in[b][k_].copy_(host_in[k_], non_blocking=True)
                    h2d_done[b][si].record(st_)
            for e_ in h2d_done[b]:
                stream.wait_event(e_)
            if i >= 2:
                for e_ in d2h_done[b]:
                    stream.wait_event(e_)                  # step i-2's outputs have been copied out
            step_into(dev_in[b], dev_outs[b])
            comp_done[b].record(stream)
            for so, st_ in enumerate(s_out):
                with torch.cuda.stream(st_):
                    st_.wait_event(comp_done[b])
                    # o, hT, dq, dk, dv, da: the three gradients on their own streams
                    for idx in ((0, 1, 2, 5), (3,), (4,))[so]:
                        host_out[b][idx].copy_(dev_outs[b][idx], non_blocking=True)
                    d2h_done[b][so].record(st_)

    e2e_run(2)
    torch.cuda.synchronize()
    barrier()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for st_ in s_in:
        st_.wait_event(f0)
    e2e_run(K)
    for st_ in s_out:
        stream.wait_stream(st_)
    f1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = replicas.max_over_ranks(f0.elapsed_time(f1) / K, world, dev)
    for code in (ws_f.read_device_status(), ws_b.read_device_status()):
        if code:
            raise RuntimeError(f"device status {code} after the timed steps")

    tokens = w.B * w.T
    value = replicas.job_throughput(tokens, world, ms)
    e2e_value = replicas.job_throughput(tokens, world, e2e_ms)
    hbm, hbm_src = peaks()
    ab = algorithmic_bytes(w, n_seq)
    dom = max((n for n in ("fwd", "bwd", "states") if n in ab), key=lambda n: kernel_ms[n])
    achieved = ab[dom] / (kernel_ms[dom] / 1000.0) / 1e9
    per_kernel = {n: {"ms": kernel_ms[n], "algorithmic_bytes": ab[n],
                      "frac": ab[n] / (kernel_ms[n] / 1000.0) / 1e9 / hbm}
                  for n in ("decay", "fwd", "states", "bwd") if n in ab and kernel_ms[n] > 0}
    abl = None
    if world == 1 and not args.no_ablation:
        abl = ablation_leg(dev)
    out = None
    if rank == 0:
        cpu = None
        if world == 1 and not args.no_cpu_baseline:
            v_, cores, desc = oracle_sample(inp, w, args.cpu_seconds)
            cpu = {"value": v_, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc}
        out = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
               "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": True,
               "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
               "config": config_of(w, world),
               "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": hbm,
                            "unit": "GB/s", "frac": achieved / hbm, "peak_source": hbm_src,
                            "traffic": measured_traffic(dom, w.name),
                            "traffic_source": traffic_source(dom, w.name),
                            "algorithmic_bytes_per_launch": ab[dom]},
               "kernel_ms": kernel_ms,
               "kernel_roofline": per_kernel,
               "ckpt": {"stride": stride, "dtype": "f32" if w.ckpt_stride else "bf16"},
               "seq_segments": seg,
               "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                       "d2h_bytes_per_step": d2h},
               "gpu_launches": launches_per_step * K,
               "clocks": clk.summary(),
               "cpu_baseline": cpu,
               "ablation": abl}
        print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()


def ablation_leg(dev, steps: int = 5, warmup: int = 3):
    """The pages' one performance claim, measured: at the 1M-token stage
    (T=1048576, H=8, dk=dv=128) one fwd+bwd step with the bounded decay (every
    diagonal tile through the tensor-core GEMMs) against the same step with the
    unbounded -softplus decay, whose diagonal tiles take the explicit
    position-pair path.  Same call sequence as the headline step (bf16 states
    handed from the forward to the backward every 128 tokens); inputs drawn
    on the device with the workloads' recipe."""
    import torch

    import chunked_linear_attention_bounded_gb300 as bdla
    from chunked_linear_attention_bounded_gb300 import bdla as B
    from chunked_linear_attention_bounded_gb300.inputs import WORKLOADS, make_inputs_on
    stream = torch.cuda.current_stream()
    res = {}
    for name in ("c1m", "c1m_ablation"):
        w = WORKLOADS[name]
        g = make_inputs_on(w, dev)
        ws_f = B.Workspace(B.workspace_bytes(B.OP_FWD, tuple(g["q"].shape), w.dv, 0, w.mode), dev)
        ws_b = B.Workspace(B.workspace_bytes(B.OP_BWD, tuple(g["q"].shape), w.dv, 0, w.mode,
                                             ckpt_stride=128), dev)
        o = torch.empty(g["v"].shape, dtype=torch.bfloat16, device=dev)
        ck = torch.empty((w.H, B.n_slots(w.B * w.T, w.B, 128), w.dk, w.dv), dtype=torch.bfloat16,
                         device=dev)
        hT = torch.empty((w.B, w.H, w.dk, w.dv), dtype=torch.float32, device=dev)
        outs = (torch.empty(g["q"].shape, dtype=torch.float32, device=dev),
                torch.empty(g["k"].shape, dtype=torch.float32, device=dev),
                torch.empty(g["v"].shape, dtype=torch.float32, device=dev),
                torch.empty(g["a"].shape, dtype=torch.float32, device=dev))

        def step():
            bdla.fwd(g["q"], g["k"], g["v"], g["a"], w.b, mode=w.mode, ws=ws_f, out=o, hT_out=hT,
                     ckpt_stride=128, ckpt_out=ck)
            bdla.bwd(g["q"], g["k"], g["v"], g["a"], g["dO"], w.b, ckpt=ck, ckpt_stride=128,
                     mode=w.mode, ws=ws_b, outs=outs)
        for _ in range(warmup):
            step()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        for code in (ws_f.read_device_status(), ws_b.read_device_status()):
            if code:
                raise RuntimeError(f"device status {code} in the {name} steps")
        res[name] = e0.elapsed_time(e1) / steps
        del g, ws_f, ws_b, o, ck, hT, outs
        torch.cuda.empty_cache()
    return {"workload": "1M-token stage, T=1048576, H=8, dk=dv=128, fwd+bwd step",
            "bounded_ms": res["c1m"], "ablation_ms": res["c1m_ablation"],
            "ablation_over_bounded": res["c1m_ablation"] / res["c1m"], "steps": steps}


def variant_arm(args, w, inp):
    """Per-channel decay (bdla_fwd_vec / bdla_bwd_vec) or the gated delta rule
    (bdla_fwd_delta / bdla_bwd_delta): one fwd+bwd step on the packed
    64K-stage documents.  Single GPU; one JSON line.  The roofline numerator
    counts the bytes the method must move: q, k, v (bf16), a (fp32: dk per
    token-head for the per-channel decay, one otherwise), beta (fp32, delta
    rule), o (bf16); backward q, k, v, dO, a, beta in and dq, dk, dv, da,
    dbeta (fp32) out.  The bf16 state before every 16-token tile, which the
    forward hands the backward, is not counted."""
    import torch

    from chunked_linear_attention_bounded_gb300 import bdla as B
    dev = torch.device("cuda", 0)
    g = {k_: (v_.to(dev) if v_ is not None else None) for k_, v_ in inp.items()}
    n_seq = (g["cu_seqlens"].numel() - 1) if g["cu_seqlens"] is not None else w.B
    nd = n_seq if g["cu_seqlens"] is not None else 0
    Dm = B.Dims(w.B, w.T, w.H, w.dk, w.dv)
    wsb = B.lib().bdla_workspace_bytes_delta if w.delta else B.lib().bdla_workspace_bytes_vec
    ws_f = B.Workspace(wsb(B.OP_FWD, Dm, nd), dev)
    ws_b = B.Workspace(wsb(B.OP_BWD, Dm, nd), dev)
    outs = [torch.empty(g["q"].shape, dtype=torch.float32, device=dev),
            torch.empty(g["k"].shape, dtype=torch.float32, device=dev),
            torch.empty(g["v"].shape, dtype=torch.float32, device=dev),
            torch.empty(g["a"].shape, dtype=torch.float32, device=dev)]
    if w.delta:
        outs.append(torch.empty(g["beta"].shape, dtype=torch.float32, device=dev))
    stream = torch.cuda.current_stream()
    # the forward hands the backward the bf16 state before every 16-token tile
    states = B.tile_states(g["q"], g["v"], g["cu_seqlens"])

    def step():
        if w.delta:
            B.fwd_delta(g["q"], g["k"], g["v"], g["a"], g["beta"], w.b, h0=g["h0"], cu_seqlens=g["cu_seqlens"],
                        mode=w.mode, ws=ws_f, states_out=states)
            B.bwd_delta(g["q"], g["k"], g["v"], g["a"], g["beta"], g["dO"], w.b, h0=g["h0"],
                        cu_seqlens=g["cu_seqlens"], mode=w.mode, ws=ws_b, outs=tuple(outs), states=states)
            return
        B.fwd_vec(g["q"], g["k"], g["v"], g["a"], w.b, h0=g["h0"], cu_seqlens=g["cu_seqlens"], mode=w.mode,
                  ws=ws_f, states_out=states)
        B.bwd_vec(g["q"], g["k"], g["v"], g["a"], g["dO"], w.b, h0=g["h0"], cu_seqlens=g["cu_seqlens"],
                  mode=w.mode, ws=ws_b, outs=tuple(outs), states=states)
    kernels = {"fwd": B.KERNEL_FWD, "bwd": B.KERNEL_BWD}
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    K = args.steps
    kev = {n: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
           for n in kernels}
    for pairs in kev.values():
        for a_, b_ in pairs:
            a_.record(stream)
            b_.record(stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with ClockSampler(0) as clk:
        e0.record(stream)
        for i in range(K):
            for n, kid in kernels.items():
                B.set_kernel_events(kid, *kev[n][i])
            step()
        e1.record(stream)
        torch.cuda.synchronize()
    for kid in kernels.values():
        B.set_kernel_events(kid, None, None)
    for code in (ws_f.read_device_status(), ws_b.read_device_status()):
        if code:
            raise RuntimeError(f"device status {code}")
    ms = e0.elapsed_time(e1) / K
    kernel_ms = {n: sum(a_.elapsed_time(b_) for a_, b_ in kev[n]) / K for n in kernels}
    th = w.B * w.T * w.H
    st = w.dk * w.dv * 4 * n_seq * w.H
    a_b = 4 * w.dk if w.vec else 4            # decay logits per token-head
    x_b = 4 if w.delta else 0                 # write strengths per token-head
    ab = {"fwd": th * (2 * w.dk * 2 + 2 * w.dv + a_b + x_b + 2 * w.dv) + 2 * st,
          "bwd": th * (2 * w.dk * 2 + 2 * w.dv * 2 + a_b + x_b + 4 * w.dk * 2 + 4 * w.dv + a_b + x_b) + st}
    hbm, hbm_src = peaks()
    dom = max(("fwd", "bwd"), key=lambda n: kernel_ms[n])
    achieved = ab[dom] / (kernel_ms[dom] / 1000.0) / 1e9
    tokens = w.B * w.T
    what = "gated delta rule" if w.delta else "per-channel decay"
    out = {"metric": f"tokens/s fwd+bwd, {what} (T=64K packed, H=32, d=128, bf16)",
           "value": tokens / (ms / 1000.0), "unit": "tokens/s", "n_gpus": 1, "steps": K,
           "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": config_of(w, 1),
           "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": hbm, "unit": "GB/s",
                        "frac": achieved / hbm, "peak_source": hbm_src, "traffic": None,
                        "algorithmic_bytes_per_launch": ab[dom]},
           "kernel_ms": kernel_ms,
           # fwd and bwd kernels, each after the document-order kernel for packed documents
           "gpu_launches": (2 + (2 if nd > 1 else 0)) * K, "clocks": clk.summary(),
           "states": "bf16 state before every 16-token tile, written by the forward, read by the backward"}
    print(json.dumps(out), flush=True)


def decode_arm(args):
    """Decode steps (bdla_decode): `--workload decode` times one new token for
    each of 256 sequences x 32 heads (dk = dv = 128) against resident fp32
    states (0.54 GB, larger than L2), a step reading and writing every state
    once.  Single GPU; prints one JSON line."""
    import torch

    from chunked_linear_attention_bounded_gb300 import bdla as B
    n_seq, H, dk, dv = 256, 32, 128, 128
    dev = torch.device("cuda", 0)
    g = torch.Generator().manual_seed(1100)
    q = (torch.randn((n_seq, H, dk), generator=g) / dk ** 0.5).bfloat16().to(dev)
    k = torch.randn((n_seq, H, dk), generator=g)
    k = (k / k.norm(dim=-1, keepdim=True)).bfloat16().to(dev)
    v = torch.randn((n_seq, H, dv), generator=g).bfloat16().to(dev)
    a = torch.randn((n_seq, H), generator=g).to(dev)
    state = (torch.randn((n_seq, H, dk, dv), generator=g) * 0.1).to(dev)
    o = torch.empty((n_seq, H, dv), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(max(3, args.warmup)):
        B.decode(q, k, v, a, state, out=o)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    K = args.steps
    with ClockSampler(0) as clk:
        e0.record(stream)
        for _ in range(K):
            B.decode(q, k, v, a, state, out=o)
        e1.record(stream)
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / K
    state_bytes = n_seq * H * dk * dv * 4
    step_bytes = 2 * state_bytes + n_seq * H * (2 * dk * 2 + 2 * dv * 2 + 4)
    hbm, hbm_src = peaks()
    achieved = step_bytes / (ms / 1000.0) / 1e9
    out = {"metric": "decode tokens/s (256 sequences x 32 heads, d=128, fp32 state)",
           "value": n_seq / (ms / 1000.0), "unit": "tokens/s", "n_gpus": 1, "steps": K,
           "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
           "config": {"workload": "decode", "sequences": n_seq, "H": H, "dk": dk, "dv": dv,
                      "l2": "state larger than L2 (%.2f GB)" % (state_bytes / 1e9)},
           "roofline": {"bound": "hbm", "kernel": "decode", "achieved": achieved, "peak": hbm,
                        "unit": "GB/s", "frac": achieved / hbm, "peak_source": hbm_src,
                        "traffic": measured_traffic("decode", "decode"),
                        "traffic_source": traffic_source("decode", "decode"),
                        "algorithmic_bytes_per_launch": step_bytes},
           "gpu_launches": K, "clocks": clk.summary()}
    print(json.dumps(out), flush=True)


def main():
    args = parse()
    if args.workload == "decode":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the decode mode has no oracle timing arm"}))
            return
        decode_arm(args)
        return
    from chunked_linear_attention_bounded_gb300.inputs import WORKLOADS, make_inputs
    import dataclasses
    rank, world, _ = dist_env()
    w = WORKLOADS[args.workload]
    if w.fwd_only:
        w = dataclasses.replace(w, fwd_only=False)
    if args.ckpt_stride is not None:
        w = dataclasses.replace(w, ckpt_stride=args.ckpt_stride)
    if args.variant is not None:
        w = dataclasses.replace(w, name=f"{w.name}_{args.variant}", vec=args.variant == "vec",
                                delta=args.variant == "delta", ckpt_stride=0)
    if args.impl == "ours":
        from chunked_linear_attention_bounded_gb300.replicas import rank_workload
        w = rank_workload(w, rank)
    if args.impl == "reference" and rank != 0:
        return
    inp = make_inputs(w, with_grad=True)
    if args.impl == "reference":
        if w.vec or w.delta:
            print(json.dumps({"impl": "reference",
                              "unavailable": "the per-channel and delta-rule modes have no oracle timing arm"}))
            return
        reference_arm(args, w, inp)
    elif w.vec or w.delta:
        variant_arm(args, w, inp)
    else:
        ours_arm(args, w, inp)


if __name__ == "__main__":
    main()
