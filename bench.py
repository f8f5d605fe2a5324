#!/usr/bin/env python
"""Throughput of the deterministic MoE layer on GB300: prints one JSON line.

A step is one pass of the whole hot path over one batch: top-k routing, schedule,
forward (gather, gate/up GEMM + SwiGLU, down GEMM + scatter, weighted reduction) and
backward (reverse-combine gather, G GEMM + SwiGLU backward + router-weight gradient,
dgrad + reverse-dispatch + k-sum, weight gradients), on the 512-expert, H=4096, I=1024,
top-10 shape with T=16384 tokens (BF16). Useful FLOPs per step: 6*R*H*I forward plus
12*R*H*I backward, R = T*K.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mok|reference]

Under torchrun (N > 1) every rank runs its own batch (weak scaling, no collective on the
data path); timing is the max over ranks. `--impl reference` times the CPU oracle on a
bounded sample of the same workload.
"""
import argparse
import hashlib
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workloads import CONFIGS, synth  # noqa: E402

METRIC = "MoE layer TFLOP/s fwd/bwd (BF16, MXFP8) on 1 GB300; % of tensor-core peak"
UNIT = "TFLOP/s"
WORKLOAD = "fwd_bf16"


# ----------------------------------------------------------------------------- helpers

def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sust=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                    src="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sust=1700.0, src="fallback")


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.f = None

    def start(self):
        try:
            self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                stderr=subprocess.DEVNULL)
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
        self.f.flush()
        rows = [r.split(",") for r in open(self.f.name).read().strip().splitlines() if r]
        os.unlink(self.f.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [c.strip() for c in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)),
                "reasons": sorted(reasons), "samples": len(sm)}


# the sources of the six tensor-core GEMM kernels (less the public header's declarations):
# the kernels whose DRAM traffic per launch profiles/ncu_traffic.json records (the ring
# forward, built on the same engine in its own file, is not among them)
GEMM_SOURCES = ("mixture_experts_layer_deterministic_gb300/csrc/gemm_tc.cu",
                "mixture_experts_layer_deterministic_gb300/csrc/gemm_pair.cu",
                "mixture_experts_layer_deterministic_gb300/csrc/gemm_tc_core.cuh",
                "mixture_experts_layer_deterministic_gb300/csrc/tc.cuh",
                "mixture_experts_layer_deterministic_gb300/csrc/common.cuh",
                "mixture_experts_layer_deterministic_gb300/csrc/mok_internal.h")


def kernel_source_sha():
    h = hashlib.sha256()
    for fn in GEMM_SOURCES:
        h.update(open(os.path.join(ROOT, fn), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel, workload):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if it was taken
    on the current kernel sources and applies to `workload` (else None)."""
    try:
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
            t = json.load(f)
        if t.get("source_sha") != kernel_source_sha() or t.get("scaled_to") != workload:
            return None
        return t["kernels"].get(kernel)
    except Exception:
        return None


# Algorithmic work of each kernel kind per call of a phase: tensor FLOPs, and the HBM bytes
# the kernel cannot avoid moving: every operand read once, every result written once, at the
# type the layer stores it (bf16 activations, pre-activations, slots and gradients; MXFP8
# operands as one byte per element plus one scale byte per 32). `used` is the number of
# experts with rows (their weights are read once per call); `save_pre` says whether the
# forward writes its pre-activations.
def algorithmic(kind, c, prec="bf16", save_pre=True, used=None):
    R, H, I, T, K = c.R, c.H, c.I, c.T, c.K
    E = c.E if used is None else used
    mx = prec == "mxfp8"
    ob = (1.0 + 1.0 / 32) if mx else 2.0        # bytes per GEMM operand element
    w13, w2 = ob * E * 2 * I * H, ob * E * H * I  # weights as the forward's GEMMs read them
    w13b, w2b = 2.0 * E * 2 * I * H, 2.0 * E * H * I  # bf16 weight-sized results (dW)
    xr, hr = ob * R * H, ob * R * I              # routed operand rows (x ring, h ring)
    row_h, row_i = 2.0 * R * H, 2.0 * R * I      # bf16 rows of width H / I
    pre = 2.0 * R * 2 * I if save_pre else 0.0   # saved pre-activations (bf16)
    flops = {"gemm_up_swiglu": 4.0 * R * H * I, "gemm_down_push": 2.0 * R * H * I,
             "ring_forward": 6.0 * R * H * I,
             "gemm_g_swiglu_bwd": 2.0 * R * H * I, "gemm_dgrad_push": 4.0 * R * H * I,
             "wgrad_w13": 4.0 * R * H * I, "wgrad_w2": 2.0 * R * H * I}
    dA_q = (1.0 + 1.0 / 32) * R * 2 * I if mx else 0.0
    hbm = {"gemm_up_swiglu": w13 + xr + hr + pre,
           "gemm_down_push": w2 + hr + row_h,                          # slots, bf16
           # dy rows, A, dA (bf16, and its MXFP8 codes) and w*h
           "gemm_g_swiglu_bwd": w2 + (ob * R * H) + 2 * row_i + 2 * row_i + row_i + dA_q,
           "gemm_dgrad_push": w13 + (dA_q if mx else 2 * row_i) + row_h,  # dx slots, bf16
           "wgrad_w13": 2.0 * R * H + 2 * row_i + w13b,
           "wgrad_w2": row_i + 2.0 * R * H + w2b,
           # the forward through a smaller ring, one launch: weights, x (read per token,
           # MXFP8 quantized), saved pre-activations and slots; h stays in the ring (L2)
           "ring_forward": w13 + w2 + ob * T * H + pre + row_h,
           "quantize_mxfp8": 2.0 * T * H + ob * T * H,
           "gather": 2.0 * T * H + xr, "combine": row_h + 2.0 * T * H + 4.0 * R,
           "dx_reduce": row_h + 2.0 * T * H, "route_topk": 4.0 * T * c.E + 8.0 * T * K,
           "gather_bwd": 2 * (2.0 * T * H) + 2 * row_h + (ob * R * H if mx else 0.0)}
    return flops.get(kind), hbm.get(kind)


# Of those bytes, the ones each kernel kind writes (the rest it reads).
def algorithmic_writes(kind, c, prec="bf16", save_pre=True, used=None):
    R, H, I, T, K = c.R, c.H, c.I, c.T, c.K
    E = c.E if used is None else used
    mx = prec == "mxfp8"
    ob = (1.0 + 1.0 / 32) if mx else 2.0
    row_h, row_i = 2.0 * R * H, 2.0 * R * I
    pre = 2.0 * R * 2 * I if save_pre else 0.0
    dA_q = (1.0 + 1.0 / 32) * R * 2 * I if mx else 0.0
    w = {"gemm_up_swiglu": ob * R * I + pre, "gemm_down_push": row_h,
         "gemm_g_swiglu_bwd": 3 * row_i + dA_q, "gemm_dgrad_push": row_h,
         "wgrad_w13": 2.0 * E * 2 * I * H, "wgrad_w2": 2.0 * E * H * I,
         "ring_forward": pre + row_h, "quantize_mxfp8": ob * T * H, "gather": ob * R * H,
         "combine": 2.0 * T * H, "dx_reduce": 2.0 * T * H, "route_topk": 8.0 * T * K,
         "gather_bwd": 2 * row_h + (ob * R * H if mx else 0.0)}
    return w.get(kind)


def measure_bandwidth(torch, dev):
    """Write-only HBM bandwidth on this GPU, now: a memset of 2 GiB, best of 5. (A read-only
    figure from a torch reduction came out below the copy bandwidth, so reads are priced at
    the copy bandwidth.)"""
    x = torch.empty(1 << 30, dtype=torch.bfloat16, device=dev)
    out = {}
    for name, fn in (("write_only_gbs", lambda: x.zero_()),):
        fn()
        best = float("inf")
        for _ in range(5):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            best = min(best, a.elapsed_time(b))
        out[name] = x.numel() * 2 / (best * 1e-3) / 1e9
    del x
    out["how"] = "torch zero_() of 2 GiB of bf16 (a memset), best of 5, CUDA events"
    return out


def roofline_of(kind, c, launches, avg_ms, pk, prec="bf16", save_pre=True, used=None):
    """Both fractions of the kernel's roofline (tensor: algorithmic FLOPs over the measured
    launch time against the dense peak of its operand type; hbm: algorithmic bytes over the
    launch time against the measured copy bandwidth), and the bound whose floor is higher,
    per launch. `launches` is the kernel's launches per call of the phase."""
    flops, nbytes = algorithmic(kind, c, prec, save_pre, used)
    if nbytes is None:
        return None
    flops = (flops or 0.0) / launches
    nbytes = nbytes / launches
    s = avg_ms * 1e-3
    tpk, tkind = pk["bf16_sust"], "bf16 sustained, " + pk["src"]
    if prec == "mxfp8" and kind not in ("wgrad_w13", "wgrad_w2"):
        tpk, tkind = 2.0 * pk["bf16_sust"], ("fp8 = 2 x bf16 sustained (the nominal dense "
                                              "ratio), " + pk["src"])
    out = {"flops_per_launch": flops, "bytes_per_launch": nbytes,
           "tflops": flops / s / 1e12, "gbs": nbytes / s / 1e9,
           "frac_tensor": flops / s / 1e12 / tpk, "frac_hbm": nbytes / s / 1e9 / pk["hbm"],
           "tensor_peak": tpk, "tensor_peak_kind": tkind}
    # a second HBM floor that also prices written bytes at the measured write-only bandwidth
    # (both terms are lower bounds on the kernel's DRAM time); reported beside the official
    # fraction
    wr = algorithmic_writes(kind, c, prec, save_pre, used)
    if wr is not None and pk.get("hbm_write"):
        wr /= launches
        floor = max(wr / (pk["hbm_write"] * 1e9), nbytes / (pk["hbm"] * 1e9))
        out["hbm_rw_floor_ms"] = floor * 1e3
        out["frac_hbm_rw"] = floor / s
    if flops / (tpk * 1e12) >= nbytes / (pk["hbm"] * 1e9):
        out.update(bound="tensor", achieved=out["tflops"], peak=tpk, unit="TFLOP/s",
                   frac=out["frac_tensor"], peak_kind=tkind, algorithmic_per_launch=flops)
    else:
        out.update(bound="hbm", achieved=out["gbs"], peak=pk["hbm"], unit="GB/s",
                   frac=out["frac_hbm"], peak_kind="hbm copy, " + pk["src"],
                   algorithmic_per_launch=nbytes)
    return out


def kernel_table(prof, calls, c, pk, prec="bf16", save_pre=True, used=None):
    """Per kernel kind from a library profile over `calls` calls of a phase: launches and
    time per call, share of the phase, and its roofline; plus the dominant kind."""
    total = max(1e-9, sum(t for _, t in prof.values()))
    table = {}
    for k, (n, t) in prof.items():
        v = {"launches_per_call": n / calls, "avg_ms": t / n, "ms_per_call": t / calls,
             "share": t / total}
        r = roofline_of(k, c, n / calls, t / n, pk, prec, save_pre, used)
        if r is not None:
            v.update(bound=r["bound"], frac=r["frac"], frac_tensor=r["frac_tensor"],
                     frac_hbm=r["frac_hbm"])
        table[k] = v
    # the dominant kernel among those with an algorithmic roofline
    ranked = sorted((k for k in prof if "bound" in table[k]), key=lambda k: -prof[k][1])
    if not ranked:
        return table, None
    dom = ranked[0]
    roof = roofline_of(dom, c, table[dom]["launches_per_call"], table[dom]["avg_ms"], pk, prec,
                       save_pre, used)
    roof["kernel"] = dom
    return table, roof


# ----------------------------------------------------------------------------- ranks

def max_over_ranks(ms, dist=None, device="cpu"):
    """The slowest rank's time: every rank runs the same number of steps on its own
    batch, so the job is done when the last rank is."""
    if dist is None:
        return ms
    import torch
    t = torch.tensor([float(ms)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(world, flops_per_rank_step, ms_max):
    """Whole-job TFLOP/s: the useful FLOPs of every rank's step over the slowest rank's
    step time (weak scaling: each rank has its own tokens)."""
    return world * flops_per_rank_step / (ms_max * 1e-3) / 1e12


def imbalanced_phases(args, torch, B, MoELayer, quantize_mxfp8, dev, w13, w2, barrier,
                      with_mx=True, profile=None):
    out = {}
    stream = torch.cuda.Stream(dev)  # a captured stream must not be the legacy default one

    def timed(fn, n):
        barrier()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n):
            fn()
        b.record(stream)
        barrier()
        return a.elapsed_time(b) / n
    for name in ("imbalanced_bf16",) + (("imbalanced_mxfp8",) if with_mx else ()):
        c = CONFIGS[name]
        mx = c.prec == "mxfp8"
        Li = MoELayer(c.T, c.H, c.I, c.E, c.K, c.minibatch, c.ring_capacity,
                      B.MOK_MXFP8 if mx else B.MOK_BF16, device=dev)
        xi = torch.from_numpy(synth.make_x(c).view(np.int16)).to(dev).view(torch.bfloat16)
        lgi = torch.from_numpy(synth.make_logits(c)).to(dev)
        if mx:
            (a13, s13), (a2, s2) = quantize_mxfp8(w13), quantize_mxfp8(w2)
        else:
            a13, s13, a2, s2 = w13, None, w2, None
        yi = torch.empty(c.T, c.H, dtype=Li.dtype, device=dev)

        def fwd_i():
            Li.route(lgi, stream)
            Li.schedule(stream=stream)
            Li.forward(xi, a13, a2, yi, s13, s2, stream=stream)
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                fwd_i()
        ms_e = timed(fwd_i, args.steps)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fwd_i()

        def replay():
            with torch.cuda.stream(stream):
                g.replay()
        replay()
        ms_g = timed(replay, args.steps)
        used = int((Li.sched.counts[:c.E] > 0).sum().item())
        out["fwd_" + name] = {"ms": ms_e, "tflops": c.fwd_flops() / (ms_e * 1e-3) / 1e12,
                              "ms_graph": ms_g,
                              "tflops_graph": c.fwd_flops() / (ms_g * 1e-3) / 1e12,
                              "tokens": c.T, "ring_rows": c.ring_capacity,
                              "experts_used": used}
        if profile is not None:
            out["fwd_" + name].update(profile(fwd_i, c, c.prec, False, used))
        del g, Li, xi, lgi, yi, a13, a2, s13, s2
        torch.cuda.empty_cache()
    return out


# ----------------------------------------------------------------------------- GPU arm

def run_mok(args):
    import torch
    from mixture_experts_layer_deterministic_gb300 import binding as B
    from mixture_experts_layer_deterministic_gb300.buffers import MoELayer, quantize_mxfp8

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    cfg = CONFIGS[args.workload]
    # weak scaling: each rank has its own tokens (seed shifted by rank), the same weights
    cfg_r = cfg.with_(seed=cfg.seed + 1000 * rank) if rank else cfg
    T, H, I, E, K = cfg.T, cfg.H, cfg.I, cfg.E, cfg.K
    R = T * K

    # pinned host inputs (the e2e leg copies these every step)
    def pinned(shape, dtype):
        return torch.empty(shape, dtype=dtype, pin_memory=True)

    hx = pinned((T, H), torch.int16)
    synth.make_x(cfg_r, out=hx.numpy().view(np.uint16))
    hdy = pinned((T, H), torch.int16)
    synth.make_dy(cfg_r, out=hdy.numpy().view(np.uint16))
    hlg = torch.from_numpy(synth.make_logits(cfg_r)).pin_memory()
    w13_host = synth.make_w13(cfg)
    w2_host = synth.make_w2(cfg)
    w13 = torch.from_numpy(w13_host.view(np.int16)).to(dev).view(torch.bfloat16)
    w2 = torch.from_numpy(w2_host.view(np.int16)).to(dev).view(torch.bfloat16)
    cpu_inputs = dict(w13=w13_host, w2=w2_host) if (rank == 0 and world == 1) else None
    if cpu_inputs is None:
        del w13_host, w2_host
    x = hx.to(dev).view(torch.bfloat16)
    dy = hdy.to(dev).view(torch.bfloat16)
    lg = hlg.to(dev)

    L = MoELayer(T, H, I, E, K, cfg.minibatch, cfg.ring_capacity, B.MOK_BF16, device=dev,
                 backward=True)
    sd = L.dtype  # outputs, saved pre-activations and weight gradients are stored as bf16
    y = torch.empty(T, H, dtype=sd, device=dev)
    pre = torch.empty(R, 2 * I, dtype=sd, device=dev)
    dx = torch.empty(T, H, dtype=sd, device=dev)
    dw13 = torch.empty(w13.shape, dtype=sd, device=dev)
    dw2 = torch.empty(w2.shape, dtype=sd, device=dev)
    dtk = torch.empty(R, dtype=torch.float32, device=dev)
    dlg = torch.empty(T, E, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def fwd():
        L.route(lg, stream)
        L.schedule(stream=stream)
        L.forward(x, w13, w2, y, saved_preact=pre, stream=stream)

    def bwd():
        L.backward(x, pre, w13, w2, dy, dx, dw13, dw2, dtk, dlg, stream=stream)

    def step():
        fwd()
        bwd()

    def barrier():
        torch.cuda.synchronize(dev)
        if dist is not None:
            dist.barrier()

    def timed(fn, n):
        barrier()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n):
            fn()
        b.record(stream)
        barrier()
        return max_over_ranks(a.elapsed_time(b) / n, dist, dev)

    for _ in range(args.warmup):
        step()
    clocks = Clocks(local)
    clocks.start()
    ms = timed(step, args.steps)
    clk = clocks.stop()
    st, dstat = B.mok_read_device_status()
    if st != B.MOK_OK or dstat != B.MOK_OK:
        raise RuntimeError("device status %d/%d" % (st, dstat))

    flops_step = cfg.fwd_flops() + cfg.bwd_flops()
    value = whole_job_value(world, flops_step, ms)

    # per-kernel timing on the launching stream over a second timed region
    pk = peaks()
    bw = measure_bandwidth(torch, dev)
    pk["hbm_write"] = bw["write_only_gbs"]
    B.check(B.mok_profile_enable(1))
    timed(step, args.steps)
    prof = B.mok_profile_read()
    B.check(B.mok_profile_enable(0))
    launches_per_step = sum(n for n, _ in prof.values()) / args.steps
    kernels, roof = kernel_table(prof, args.steps, cfg, pk)
    tr = ncu_traffic(roof["kernel"], args.workload)
    roof["traffic"] = tr
    if tr is not None:
        roof["traffic_over_algorithmic"] = tr / roof["bytes_per_launch"]
    # DRAM traffic of every GEMM against its algorithmic bytes, where the committed ncu
    # summary applies to these kernel sources
    for k, v in kernels.items():
        t = ncu_traffic(k, args.workload)
        r = roofline_of(k, cfg, v["launches_per_call"], v["avg_ms"], pk)
        if t is not None and r is not None:
            v["traffic_over_algorithmic"] = t / r["bytes_per_launch"]

    def profile(fn, c, prec, save_pre, used=None):
        """per-kernel table and dominant-kernel roofline of a phase (library events on the
        launching stream over args.steps calls)"""
        B.check(B.mok_profile_enable(1))
        timed(fn, args.steps)
        pr = B.mok_profile_read()
        B.check(B.mok_profile_enable(0))
        table, rf = kernel_table(pr, args.steps, c, pk, prec, save_pre, used)
        return {"kernels": {k: {kk: (round(vv, 5) if isinstance(vv, float) else vv)
                                for kk, vv in v.items()} for k, v in table.items()},
                "roofline": rf}

    # phases: forward alone, backward alone, MXFP8 forward
    phases = {}
    ms_f = timed(fwd, args.steps)
    phases["fwd_bf16"] = {"ms": ms_f, "tflops": cfg.fwd_flops() / (ms_f * 1e-3) / 1e12}
    ms_b = timed(bwd, args.steps)
    phases["bwd_bf16"] = {"ms": ms_b, "tflops": cfg.bwd_flops() / (ms_b * 1e-3) / 1e12,
                          "tokens": T}

    # the BF16 backward workload (T = 8192, its own seeded inputs), after a forward that
    # saved its pre-activations
    if not args.no_bwd8k:
        cb = CONFIGS["bwd_bf16"]
        Lb = MoELayer(cb.T, H, I, E, K, cb.minibatch, cb.ring_capacity, B.MOK_BF16, device=dev,
                      backward=True)
        xb = torch.from_numpy(synth.make_x(cb).view(np.int16)).to(dev).view(torch.bfloat16)
        dyb = torch.from_numpy(synth.make_dy(cb).view(np.int16)).to(dev).view(torch.bfloat16)
        Rb = cb.T * K
        preb = torch.empty(Rb, 2 * I, dtype=sd, device=dev)
        yb, dxb = torch.empty(cb.T, H, dtype=sd, device=dev), torch.empty(cb.T, H, dtype=sd,
                                                                             device=dev)
        dtkb = torch.empty(Rb, dtype=torch.float32, device=dev)
        dlgb = torch.empty(cb.T, E, dtype=torch.float32, device=dev)
        Lb.route(torch.from_numpy(synth.make_logits(cb)).to(dev), stream)
        Lb.schedule(stream=stream)
        Lb.forward(xb, w13, w2, yb, saved_preact=preb, stream=stream)

        def bwd8k():
            Lb.backward(xb, preb, w13, w2, dyb, dxb, dw13, dw2, dtkb, dlgb, stream=stream)
        for _ in range(2):
            bwd8k()
        ms_b8 = timed(bwd8k, args.steps)
        phases["bwd_bf16_T8192"] = {"ms": ms_b8, "tokens": cb.T,
                                    "tflops": cb.bwd_flops() / (ms_b8 * 1e-3) / 1e12}
        phases["bwd_bf16_T8192"].update(profile(bwd8k, cb, "bf16", True))
        del Lb, xb, dyb, preb, yb, dxb, dtkb, dlgb
        torch.cuda.empty_cache()

    # backward without saved pre-activations: the gate/up GEMM is recomputed inside it
    # (its FLOPs are not useful work and are not counted)
    def bwd_rc():
        L.backward(x, None, w13, w2, dy, dx, dw13, dw2, dtk, dlg, stream=stream)
    bwd_rc()
    ms_r = timed(bwd_rc, args.steps)
    phases["bwd_bf16_recompute"] = {"ms": ms_r,
                                    "tflops": cfg.bwd_flops() / (ms_r * 1e-3) / 1e12}

    # the shared expert's forward (every token, weight one), added into y
    from mixture_experts_layer_deterministic_gb300.buffers import SharedExpert
    S = SharedExpert(L)
    w13s = (torch.randn(2 * I, H, device=dev) * cfg.w_std).to(torch.bfloat16)
    w2s = (torch.randn(H, I, device=dev) * cfg.w_std).to(torch.bfloat16)

    def fwd_shared():
        S.forward(x, w13s, w2s, y, stream=stream)
    fwd_shared()
    ms_s = timed(fwd_shared, args.steps)
    phases["fwd_shared_bf16"] = {"ms": ms_s, "tflops": 6.0 * T * H * I / (ms_s * 1e-3) / 1e12}

    # and its backward (dx += its input gradient, its weight gradients), after a forward
    # that saved its pre-activations
    pre_s = torch.empty(T, 2 * I, dtype=sd, device=dev)
    dw13s = torch.empty(2 * I, H, dtype=sd, device=dev)
    dw2s = torch.empty(H, I, dtype=sd, device=dev)
    S.forward(x, w13s, w2s, y, saved_preact=pre_s, stream=stream)

    def bwd_shared():
        S.backward(x, w13s, w2s, pre_s, dy, dx, dw13s, dw2s, stream=stream)
    bwd_shared()
    ms_sb = timed(bwd_shared, args.steps)
    phases["bwd_shared_bf16"] = {"ms": ms_sb,
                                 "tflops": 12.0 * T * H * I / (ms_sb * 1e-3) / 1e12}
    del S, w13s, w2s, pre_s, dw13s, dw2s

    # the imbalanced workload's forward (Zipf-skewed routing, 65536 tokens, a ring of 2960
    # rows, so many passes): eager, and replayed from a captured CUDA graph
    if not args.no_imbalanced:
        phases.update(imbalanced_phases(args, torch, B, MoELayer, quantize_mxfp8, dev, w13, w2,
                                        barrier, with_mx=not args.no_mxfp8, profile=profile))
    if not args.no_mxfp8:
        q13, s13 = quantize_mxfp8(w13)
        q2, s2 = quantize_mxfp8(w2)
        Lm = MoELayer(T, H, I, E, K, cfg.minibatch, cfg.ring_capacity, B.MOK_MXFP8, device=dev)

        def fwd_mx():
            Lm.route(lg, stream)
            Lm.schedule(stream=stream)
            Lm.forward(x, q13, q2, y, s13, s2, stream=stream)

        for _ in range(2):
            fwd_mx()
        ms_m = timed(fwd_mx, args.steps)
        phases["fwd_mxfp8"] = {"ms": ms_m, "tflops": cfg.fwd_flops() / (ms_m * 1e-3) / 1e12}
        phases["fwd_mxfp8"].update(profile(fwd_mx, cfg, "mxfp8", False))

        # the shared expert's MXFP8 forward on weights quantized once (untimed), added into y
        from mixture_experts_layer_deterministic_gb300.buffers import SharedExpert
        Sm = SharedExpert(Lm)
        ws13 = quantize_mxfp8((torch.randn(2 * I, H, device=dev) * cfg.w_std).to(torch.bfloat16))
        ws2 = quantize_mxfp8((torch.randn(H, I, device=dev) * cfg.w_std).to(torch.bfloat16))

        def fwd_shared_mx():
            Sm.forward(x, ws13, ws2, y, stream=stream)
        fwd_shared_mx()
        ms_sm = timed(fwd_shared_mx, args.steps)
        phases["fwd_shared_mxfp8"] = {"ms": ms_sm,
                                      "tflops": 6.0 * T * H * I / (ms_sm * 1e-3) / 1e12}
        # and its MXFP8 backward on the transposed quantized weights (untimed), after a
        # forward that saved its pre-activations
        from mixture_experts_layer_deterministic_gb300.buffers import quantize_mxfp8_transposed
        w13s_b = (torch.randn(1, 2 * I, H, device=dev) * cfg.w_std).to(torch.bfloat16)
        w2s_b = (torch.randn(1, H, I, device=dev) * cfg.w_std).to(torch.bfloat16)
        ws13, ws2 = quantize_mxfp8(w13s_b[0]), quantize_mxfp8(w2s_b[0])
        wst13, wst2 = quantize_mxfp8_transposed(w13s_b), quantize_mxfp8_transposed(w2s_b)
        pre_s = torch.empty(T, 2 * I, dtype=sd, device=dev)
        dw13s = torch.empty(2 * I, H, dtype=sd, device=dev)
        dw2s = torch.empty(H, I, dtype=sd, device=dev)
        Sm.forward(x, ws13, ws2, y, saved_preact=pre_s, stream=stream)

        def bwd_shared_mx():
            Sm.backward(x, wst13, wst2, pre_s, dy, dx, dw13s, dw2s, stream=stream)
        bwd_shared_mx()
        ms_smb = timed(bwd_shared_mx, args.steps)
        phases["bwd_shared_mxfp8"] = {"ms": ms_smb,
                                      "tflops": 12.0 * T * H * I / (ms_smb * 1e-3) / 1e12}
        del Sm, ws13, ws2, w13s_b, w2s_b, wst13, wst2, pre_s, dw13s, dw2s

        # MXFP8 backward (G and dgrad in MXFP8 on weights pre-quantized along their
        # contraction axes, untimed like the forward's; weight gradients BF16), after an
        # MXFP8 forward that saved its pre-activations
        from mixture_experts_layer_deterministic_gb300.buffers import (
            backward_mxfp8, quantize_mxfp8_transposed)
        w13t, w2t = quantize_mxfp8_transposed(w13), quantize_mxfp8_transposed(w2)
        Lm.route(lg, stream)
        Lm.schedule(stream=stream)
        Lm.forward(x, q13, q2, y, s13, s2, saved_preact=pre, stream=stream)

        def bwd_mx():
            backward_mxfp8(Lm, x, pre, w13t, w2t, dy, dx, dw13, dw2, dtk, dlg, stream=stream)
        for _ in range(2):
            bwd_mx()
        ms_mb = timed(bwd_mx, args.steps)
        phases["bwd_mxfp8"] = {"ms": ms_mb, "tflops": cfg.bwd_flops() / (ms_mb * 1e-3) / 1e12}
        phases["bwd_mxfp8"].update(profile(bwd_mx, cfg, "mxfp8", True))
        del Lm, q13, s13, q2, s2, w13t, w2t

    # e2e through the public API with host buffers: every step copies its inputs (x, logits,
    # dy) from pinned host memory and reads its results (y, dx) back. As a training loop
    # prefetches its next batch, the copies run on their own streams: the H2D of step i+1
    # overlaps step i's kernels, dy is waited for only by the backward, y is read back
    # while the backward runs and dx during the next step, with double-buffered device
    # inputs and outputs ordered by events. The first H2D and the last D2H are inside the
    # timed region.
    hy = pinned((T, H), torch.int16)   # bf16 outputs
    hdx = pinned((T, H), torch.int16)
    xin = [x, torch.empty_like(x)]
    lgin = [lg, torch.empty_like(lg)]
    dyin = [dy, torch.empty_like(dy)]
    yout = [y, torch.empty_like(y)]
    dxout = [dx, torch.empty_like(dx)]
    h2d_s = torch.cuda.Stream(dev)
    d2h_s = torch.cuda.Stream(dev)

    def e2e_run(n):
        ev_in_f = [torch.cuda.Event() for _ in range(2)]  # x, logits of buffer b have landed
        ev_in_b = [torch.cuda.Event() for _ in range(2)]  # dy of buffer b has landed
        ev_fwd = [torch.cuda.Event() for _ in range(2)]   # the forward on buffer b is done
        ev_used = [torch.cuda.Event() for _ in range(2)]  # the step on buffer b is done
        ev_out = [torch.cuda.Event() for _ in range(2)]   # outputs of buffer b are on host
        barrier()
        a = torch.cuda.Event(enable_timing=True)
        b_ = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        h2d_s.wait_event(a)

        def h2d(i):
            b = i % 2
            with torch.cuda.stream(h2d_s):
                h2d_s.wait_event(ev_used[b])  # step i-2 has finished with buffer b
                xin[b].view(torch.int16).copy_(hx, non_blocking=True)
                lgin[b].copy_(hlg, non_blocking=True)
                ev_in_f[b].record(h2d_s)
                dyin[b].view(torch.int16).copy_(hdy, non_blocking=True)  # needed by the bwd
                ev_in_b[b].record(h2d_s)

        h2d(0)
        for i in range(n):
            b = i % 2
            if i + 1 < n:
                h2d(i + 1)
            stream.wait_event(ev_in_f[b])
            stream.wait_event(ev_out[b])  # the D2H of step i-2 has read outputs b
            L.route(lgin[b], stream)
            L.schedule(stream=stream)
            L.forward(xin[b], w13, w2, yout[b], saved_preact=pre, stream=stream)
            ev_fwd[b].record(stream)
            with torch.cuda.stream(d2h_s):  # y leaves while the backward runs
                d2h_s.wait_event(ev_fwd[b])
                hy.copy_(yout[b].view(torch.int16), non_blocking=True)
            stream.wait_event(ev_in_b[b])
            L.backward(xin[b], pre, w13, w2, dyin[b], dxout[b], dw13, dw2, dtk, dlg,
                       stream=stream)
            ev_used[b].record(stream)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(ev_used[b])
                hdx.copy_(dxout[b].view(torch.int16), non_blocking=True)
                ev_out[b].record(d2h_s)
        stream.wait_event(ev_out[(n - 1) % 2])
        b_.record(stream)
        barrier()
        return max_over_ranks(a.elapsed_time(b_) / n, dist, dev)

    e2e_run(2)
    ms_e = e2e_run(args.steps)
    h2d = hx.numel() * 2 + hlg.numel() * 4 + hdy.numel() * 2
    d2h = hy.numel() * 2 + hdx.numel() * 2

    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded Gaussian)",
        "config": {"workload": "fwd+bwd BF16, %d experts, H=%d, I=%d, top-%d, T=%d" % (
                       E, H, I, K, T),
                   "T": T, "H": H, "I": I, "E": E, "K": K, "minibatch": cfg.minibatch,
                   "ring_capacity": cfg.ring_capacity or "all rows",
                   "l2": "inputs larger than L2 (%.1f GB of "
                   "expert weights read per step)" % (3.0 * E * H * I * 2 / 1e9),
                   "parallelism": "replicas" if world > 1
                   else "single GPU"},
        "e2e": {"value": whole_job_value(world, flops_step, ms_e), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms_e},
        "gpu_launches": int(round(launches_per_step * args.steps)),
        "roofline": roof,
        "phases": phases,
        "kernels": {k: {kk: (round(vv, 5) if isinstance(vv, float) else vv)
                        for kk, vv in v.items()} for k, v in kernels.items()},
        "clocks": clk,
        "peaks": pk,
        "bandwidth": bw,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(cfg, cpu_inputs, budget_s=args.cpu_seconds)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# ----------------------------------------------------------------------------- CPU oracle

def oracle_sample(cfg, host, n_tokens, n_experts):
    """Times the oracle on a bounded sample: the forward of n_tokens tokens (with all their
    K experts) and the backward of every routed row of n_experts experts. Returns
    (useful FLOPs, seconds, description)."""
    import oracle
    lg = synth.make_logits(cfg)
    idx, w = oracle.route(lg.astype(np.float64), cfg.K)
    x = host.get("x")
    if x is None:
        x = synth.make_x(cfg)
    toks = np.arange(n_tokens)
    idx_s = idx[toks]
    used = np.unique(idx_s)
    remap = np.full(cfg.E, -1, np.int32)
    remap[used] = np.arange(len(used), dtype=np.int32)
    w13, w2 = host["w13"], host["w2"]
    t0 = time.perf_counter()
    oracle.forward(oracle.bf16_to_f64(x[toks]), remap[idx_s], w[toks], w13[used], w2[used],
                   mode=oracle.BF16)
    t_fwd = time.perf_counter() - t0
    flops = 6.0 * n_tokens * cfg.K * cfg.H * cfg.I
    dy = synth.make_dy(cfg)
    t_bwd = 0.0
    rows = 0
    for e in range(n_experts):
        t_e, k_e = np.nonzero(idx == e)
        t0 = time.perf_counter()
        oracle.backward(oracle.bf16_to_f64(x[t_e]), np.zeros((len(t_e), 1), np.int32),
                        w[t_e, k_e][:, None], w13[e:e + 1], w2[e:e + 1],
                        oracle.bf16_to_f64(dy[t_e]), mode=oracle.BF16)
        t_bwd += time.perf_counter() - t0
        rows += len(t_e)
    flops += 12.0 * rows * cfg.H * cfg.I
    desc = ("forward of %d tokens (%d routed rows) + backward of all %d routed rows of "
            "experts 0..%d" % (n_tokens, n_tokens * cfg.K, rows, n_experts - 1))
    return flops, t_fwd + t_bwd, desc


def cores():
    n = os.environ.get("OMP_NUM_THREADS")
    return int(n) if n else (os.cpu_count() or 1)


def cpu_baseline(cfg, host, budget_s=20.0):
    flops, sec, desc = oracle_sample(cfg, host, 8, 1)   # calibration
    rate = flops / sec
    # size the sample to about budget_s seconds
    n_tok = int(max(8, min(cfg.T, 8 * budget_s / 2 / max(sec, 1e-3))))
    n_exp = int(max(1, min(cfg.E, budget_s / 2 / max(sec, 1e-3))))
    flops, sec, desc = oracle_sample(cfg, host, n_tok, n_exp)
    return {"value": flops / sec / 1e12, "unit": UNIT, "cores": cores(), "kind": "oracle",
            "sample": desc, "seconds": sec, "calibration_tflops": rate / 1e12}


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    cfg = CONFIGS[args.workload]
    host = dict(w13=synth.make_w13(cfg), w2=synth.make_w2(cfg), x=synth.make_x(cfg))
    n_tok, n_exp = args.ref_tokens, args.ref_experts
    for _ in range(args.warmup):
        oracle_sample(cfg, host, n_tok, n_exp)
    tot_f, tot_s, desc = 0.0, 0.0, ""
    for _ in range(args.steps):
        f, s, desc = oracle_sample(cfg, host, n_tok, n_exp)
        tot_f += f
        tot_s += s
    value = tot_f / tot_s / 1e12
    out = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": tot_s / args.steps * 1e3,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (seeded Gaussian)", "impl": "reference",
           "config": {"workload": "fwd+bwd BF16, 512 experts, H=4096, I=1024, top-10, "
                                  "T=16384 (bounded sample per step)"},
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores(), "kind": "oracle",
                            "sample": desc},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="mok", choices=["mok", "reference"])
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(CONFIGS))
    ap.add_argument("--no-mxfp8", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-imbalanced", action="store_true")
    ap.add_argument("--no-bwd8k", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=20.0)
    ap.add_argument("--ref-tokens", type=int, default=16)
    ap.add_argument("--ref-experts", type=int, default=1)
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "mok":
        args.warmup = 3
    return args


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_mok(args)


if __name__ == "__main__":
    main()
