#!/usr/bin/env python3
"""Benchmark of the chunkwise causal linear attention forward pass on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--C C]
                    [--impl ours|reference] [--path auto|simt|tc]

One step = one la_chunked_fwd call over the whole workload (feature map, chunk states,
chunk scan, intra/inter outputs, normaliser, store).  Default workload: elu+1 features
with the normaliser, B=8 H=16 L=8192 d_k=d_v=128, bf16, C=64 (the L=8192, d=128 case the
throughput target is stated on).  Prints one JSON line on rank 0.

Multi-GPU (torchrun): (b, h) heads are independent problems, so every rank runs its own
copy of the workload (weak scaling, no collective on the data path); the barrier and the
max over ranks only frame the timing.

--impl reference times the CPU oracle (chunk-size-1 recurrence, fp64) on the host cores,
each step a bounded sample of heads of the same workload.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

L2_BYTES = 126 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
METRIC = "tokens/sec (B·H·L/s) chunked causal linear-attn fwd; % of bf16 TC roofline"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="elu1-norm-d128-L8192", choices=list(synth.WORKLOADS))
    ap.add_argument("--C", type=int, default=None)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--path", default="auto", choices=["auto", "simt", "tc"])
    ap.add_argument("--seed", type=int, default=11)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--B", type=int, default=None, help="override the workload's batch")
    ap.add_argument("--H", type=int, default=None, help="override the workload's heads")
    ap.add_argument("--L", type=int, default=None,
                    help="override the workload's sequence length (profiling captures)")
    ap.add_argument("--op", default="forward",
                    choices=["forward", "decode", "noncausal", "backward"],
                    help="forward: the chunked forward (the headline metric); decode: one "
                         "la_decode_step per step for every head of the workload; noncausal: "
                         "la_noncausal_fwd over the workload (bidirectional); backward: "
                         "la_chunked_bwd over the workload")
    return ap.parse_args()


def max_over_ranks(dist, value, device="cpu"):
    """The largest `value` over all ranks (the job is as slow as its slowest rank)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world, units_per_rank_step, steps, max_ms):
    """Whole-job units per second under weak scaling: every rank runs its own copy of the
    workload, so the job processes world x units per step in the slowest rank's time."""
    return world * units_per_rank_step * steps / (max_ms / 1e3)


def workload_config(name, w, C):
    return {"workload": name, "B": w["B"], "H": w["H"], "L": w["L"], "dk": w["dk"],
            "dv": w["dv"], "C": C, "feature_map": w["fm"], "m": w["m"],
            "normalize": bool(w["normalize"]), "loglinear": bool(w.get("loglinear")),
            "storage": w["dtype"], **({"gamma": w["gamma"]} if w.get("gamma") else {})}


def bytes_per_token(w):
    es = 2 if w["dtype"] == "bf16" else 4
    b = es * (2 * w["dk"] + 2 * w["dv"])
    if w.get("loglinear"):
        b += 4 * synth.num_levels(w["L"])
    return b


def flops_per_token(w, C):
    """Chunked-order FLOPs per token: 2x the chunked page's multiply-add counts
    (state write + read 2 D dv, scores + value mixing C (D + dv)) plus the FAVOR+
    projection of q and k (2 * 2 dk m)."""
    D = w["m"] if w["fm"] == "favor" else w["dk"]
    f = 2 * (2 * D * w["dv"] + C * (D + w["dv"]))
    if w["fm"] == "favor":
        f += 2 * 2 * w["dk"] * w["m"]
    return f


def kernel_sha1(w, C=64):
    """Hash of the tensor-core kernel source that serves workload `w` at chunk size C (plus
    the shared headers): a committed DRAM-traffic figure is only used while this is
    unchanged."""
    import hashlib
    d = os.path.join(ROOT, "chunkwise_causal_linear_gb300", "csrc")
    if w.get("loglinear"):
        main = "tc_loglinear.cu"
    elif w["fm"] == "favor":
        main = "tc_favor.cu"
    elif C > 64:
        main = "tc_wide.cu"
    else:
        main = "tc.cu"
    h = hashlib.sha1()
    for name in (main, "tc_ptx.cuh", "tc_common.cuh"):
        with open(os.path.join(d, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def ncu_traffic(workload, C, path, B, H, L=None):
    """DRAM bytes per launch from the committed ncu capture (profiles/traffic.json), or None
    when there is none for this workload or the kernel changed since it was taken."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f).get(f"{workload}/C{C}/{path}")
    except Exception:
        return None
    w = synth.WORKLOADS[workload]
    if not rec or rec.get("kernel_sha1") != kernel_sha1(w, C) or (B, H) != (w["B"], w["H"]):
        return None
    if L is not None and L != w["L"]:
        return None
    return rec["bytes_per_launch"]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return json.load(f), "measured"
    except Exception:
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": 1900.0}, "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled in the background."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu)], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        sms, maxes, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sms.append(float(f[1]))
                maxes.append(float(f[2]))
            except ValueError:
                continue
            for n, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        if not sms:
            return None
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxes),
                "reasons": sorted(reasons), "samples": len(sms)}


def cpu_baseline(w, inp_heads, heads_used, threads):
    """Times the oracle's chunk-size-1 recurrence (Fenwick recurrence for the log-linear
    mask) on the given heads, one head per host thread."""
    import oracle
    q = synth.as_f64(inp_heads["q"], w["dtype"])
    k = synth.as_f64(inp_heads["k"], w["dtype"])
    v = synth.as_f64(inp_heads["v"], w["dtype"])
    lam = None if inp_heads["lam"] is None else inp_heads["lam"].astype(np.float64)
    om = None if inp_heads["omega"] is None else inp_heads["omega"].astype(np.float64)
    oracle.lib()
    t0 = time.perf_counter()
    oracle.forward(q, k, v, fm=w["fm"], omega=om, normalize=w["normalize"], lam=lam,
                   method="recurrence", threads=threads, gamma=w.get("gamma"))
    dt = time.perf_counter() - t0
    toks = heads_used * w["L"]
    return toks / dt, dt


def cpu_baseline_one_core(w, inp_heads):
    """The same oracle recurrence on one head, one thread: the single-core rate."""
    one = {kk: (vv[:1] if kk in ("q", "k", "v", "lam") and vv is not None else vv)
           for kk, vv in inp_heads.items()}
    val, dt = cpu_baseline(w, one, 1, 1)
    return {"value": val, "unit": "tokens/s", "cores": 1,
            "sample": f"1 head x L={w['L']}, {dt:.2f} s wall"}


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def oracle_flops_per_token(w):
    """FLOPs per token of the oracle's chunk-size-1 recurrence (state update + read, one
    state per Fenwick level for the log-linear mask, plus the FAVOR+ projections)."""
    D = w["m"] if w["fm"] == "favor" else w["dk"]
    n_states = synth.num_levels(w["L"]) if w.get("loglinear") else 1
    f = 2 * D * w["dv"] * (1 + n_states)
    if w["fm"] == "favor":
        f += 2 * 2 * w["dk"] * w["m"]
    return f


def sample_heads(w, cores, core_seconds=20.0, flops_per_core=2.5e9):
    """A bounded sample of heads: about `core_seconds` of oracle work on the host cores,
    at least one head per core when that is cheaper, at most all heads."""
    n = w["B"] * w["H"]
    per_head = w["L"] * oracle_flops_per_token(w) / flops_per_core
    want = int(core_seconds // max(per_head, 1e-9))
    want = max(1, min(n, max(want, min(cores, n)) if per_head * cores < core_seconds else want))
    return list(range(want))


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    w = dict(synth.WORKLOADS[args.workload])
    if args.B:
        w["B"] = args.B
    if args.H:
        w["H"] = args.H
    if args.L:
        w["L"] = args.L
    C = args.C if args.C is not None else w["C"]
    cores = host_cores()
    heads = sample_heads(w, cores)
    inp = synth.make_inputs(w, args.seed, heads=heads)
    for _ in range(max(0, args.warmup)):
        cpu_baseline(w, inp, len(heads), cores)
        break  # one warm-up pass is enough for a CPU loop; the rest would only burn time
    times = []
    for _ in range(args.steps):
        _, dt = cpu_baseline(w, inp, len(heads), cores)
        times.append(dt)
    tot = sum(times)
    value = args.steps * len(heads) * w["L"] / tot
    sample = f"{len(heads)} of {w['B'] * w['H']} heads x L={w['L']} per step"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * tot / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(args.workload, w, C),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores,
                             "kind": "oracle", "sample": sample,
                             "one_core": cpu_baseline_one_core(w, inp)},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import torch

    import chunkwise_causal_linear_gb300 as la
    from chunkwise_causal_linear_gb300 import build as la_build

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    if rank == 0 or not la_build.up_to_date():
        la_build.build()
    if dist:
        dist.barrier()

    w = dict(synth.WORKLOADS[args.workload])
    if args.B:
        w["B"] = args.B
    if args.H:
        w["H"] = args.H
    if args.L:
        w["L"] = args.L
    C = args.C if args.C is not None else w["C"]
    B, H, L, dk, dv = w["B"], w["H"], w["L"], w["dk"], w["dv"]
    path = {"auto": la.LA_PATH_AUTO, "simt": la.LA_PATH_SIMT, "tc": la.LA_PATH_TC}[args.path]
    dtype = la.LA_BF16 if w["dtype"] == "bf16" else la.LA_F32
    tdt = torch.bfloat16 if w["dtype"] == "bf16" else torch.float32

    inp = synth.make_inputs(w, args.seed)

    def host_tensor(x, shape):
        if w["dtype"] == "bf16":
            t = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16)
        else:
            t = torch.from_numpy(x)
        return t.reshape(shape).pin_memory()

    qh, kh, vh = (host_tensor(inp["q"], (B, H, L, dk)), host_tensor(inp["k"], (B, H, L, dk)),
                  host_tensor(inp["v"], (B, H, L, dv)))
    q, k, v = qh.cuda(), kh.cuda(), vh.cuda()
    out = torch.empty((B, H, L, dv), dtype=tdt, device="cuda")
    outh = torch.empty((B, H, L, dv), dtype=tdt).pin_memory()
    omega = None if inp["omega"] is None else torch.from_numpy(inp["omega"]).cuda()
    lam = None if inp["lam"] is None else torch.from_numpy(inp["lam"]).reshape(
        B, H, L, -1).cuda()
    nl = 0 if lam is None else lam.shape[-1]
    fm = la.make_feature_map(w["fm"], w["m"], omega.data_ptr() if omega is not None else 0)
    gamma = w.get("gamma")  # Retention decay: la_decay_fwd
    if gamma is not None and args.op != "forward":
        raise SystemExit("decay workloads: --op forward only")
    if gamma is None:
        wsb = la.la_chunked_workspace_bytes(B, H, L, dk, dv, C, fm, int(w["normalize"]), nl, dtype)
        rc, plan = la.la_chunked_plan(B, H, L, dk, dv, C, fm, int(w["normalize"]),
                                      int(lam is not None), nl, dtype, path, 0)
    else:
        wsb = la.la_decay_workspace_bytes(B, H, L, dk, dv, C, fm, int(w["normalize"]), gamma, dtype)
        rc, plan = la.la_decay_plan(B, H, L, dk, dv, C, fm, int(w["normalize"]), gamma, dtype, path)
    ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device="cuda")
    if rc != la.LA_OK:
        raise la.LAError(rc, "plan")
    stream = torch.cuda.current_stream()
    sptr = stream.cuda_stream
    lam_ptr = lam.data_ptr() if lam is not None else None
    noncausal = args.op == "noncausal"
    if noncausal:
        if lam is not None:
            raise SystemExit("--op noncausal: the log-linear mask is causal")
        wsb = la.la_noncausal_workspace_bytes(B, H, L, dk, dv, fm, int(w["normalize"]), dtype)
        if wsb == 0:
            raise SystemExit("--op noncausal: unsupported sizes")
        ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
        # two launches on either path: the per-head state, then the outputs
        plan = dict(plan, n_launches=2, path="noncausal")

    def step():
        if noncausal:
            r = la.la_noncausal_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, H,
                                    L, dk, dv, fm, int(w["normalize"]), dtype, ws.data_ptr(), wsb,
                                    sptr)
        elif gamma is not None:
            r = la.la_decay_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, H, L,
                                dk, dv, C, fm, int(w["normalize"]), gamma, dtype, ws.data_ptr(),
                                wsb, sptr, path)
        else:
            r = la.la_chunked_fwd_path(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B,
                                       H, L, dk, dv, C, fm, int(w["normalize"]), lam_ptr, nl, dtype,
                                       ws.data_ptr(), wsb, sptr, path)
        if r != la.LA_OK:
            raise la.LAError(r, "la_noncausal_fwd" if noncausal else "la_chunked_fwd")

    io_bytes = B * H * L * bytes_per_token(w)
    flush = None
    if io_bytes < 2 * L2_BYTES:
        flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device="cuda")

    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize()
    st = la.la_last_device_status(sptr)
    if st != la.LA_OK:
        raise la.LAError(st, "device status after warm-up")

    clocks = ClockSampler(torch.cuda.current_device())
    if rank == 0:
        clocks.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for i in range(args.steps):
        if flush is not None:
            flush.zero_()
        evs[i][0].record(stream)
        step()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clk = clocks.stop() if rank == 0 else None
    times = [a.elapsed_time(b) for a, b in evs]
    t_ms = sum(times)
    st = la.la_last_device_status(sptr)
    if st != la.LA_OK:
        raise la.LAError(st, "device status after the timed steps")
    t_ms = max_over_ranks(dist, t_ms, "cuda")

    tokens_per_step = B * H * L
    value = job_throughput(world, tokens_per_step, args.steps, t_ms)
    ms_per_step = t_ms / args.steps

    # ---- end to end through the host-buffer entry point (copies inside the region)
    e2e = None
    if not args.no_e2e and not noncausal:
        h2d = int(qh.numel() * qh.element_size() * 2 + vh.numel() * vh.element_size())
        d2h = int(outh.numel() * outh.element_size())
        qd, kd, vd = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

        def e2e_step():
            if gamma is not None:
                # no host-buffer entry point for the decay: the same copies, queued around it
                qd.copy_(qh, non_blocking=True)
                kd.copy_(kh, non_blocking=True)
                vd.copy_(vh, non_blocking=True)
                r = la.la_decay_fwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), out.data_ptr(), B,
                                    H, L, dk, dv, C, fm, int(w["normalize"]), gamma, dtype,
                                    ws.data_ptr(), wsb, sptr, path)
                if r != la.LA_OK:
                    raise la.LAError(r, "la_decay_fwd")
                outh.copy_(out, non_blocking=True)
                return
            r = la.la_chunked_fwd_host(qh.data_ptr(), kh.data_ptr(), vh.data_ptr(),
                                       outh.data_ptr(), qd.data_ptr(), kd.data_ptr(),
                                       vd.data_ptr(), out.data_ptr(), B, H, L, dk, dv, C, fm,
                                       int(w["normalize"]), lam_ptr, nl, dtype, ws.data_ptr(),
                                       wsb, sptr)
            if r != la.LA_OK:
                raise la.LAError(r, "la_chunked_fwd_host")

        for _ in range(max(1, min(args.warmup, 3))):
            e2e_step()
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n_e2e = max(1, min(args.steps, 10))
        e0.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        te = max_over_ranks(dist, e0.elapsed_time(e1), "cuda")
        e2e = {"value": job_throughput(world, tokens_per_step, n_e2e, te), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n_e2e}

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0

    peaks, peak_kind = measured_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    tpk = float(peaks.get("bf16_tflops", FALLBACK_BF16_TFLOPS))
    kernel_s = (t_ms / args.steps) / 1e3
    flops = tokens_per_step * flops_per_token(w, C)
    traffic = ncu_traffic(args.workload, C, plan["path"], B, H, L)
    # the binding roofline is the one with the longer ideal time: HBM bytes at the copy
    # bandwidth, or the chunked order's FLOPs at the bf16 tensor rate (a kernel timed
    # alone: the burst figure)
    tensor_bound = flops / (tpk * 1e12) > io_bytes / (hbm * 1e9)
    if tensor_bound:
        achieved = flops / kernel_s / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": tpk, "unit": "TFLOP/s",
                "frac": achieved / tpk, "traffic": traffic,
                "peak_kind": f"{peak_kind} bf16_tflops (cuBLAS burst)",
                "algorithmic_flops_per_launch": flops, "algorithmic_bytes_per_launch": io_bytes,
                "hbm_gbs": io_bytes / kernel_s / 1e9, "hbm_peak_gbs": hbm}
    else:
        achieved = io_bytes / kernel_s / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm, "traffic": traffic,
                "peak_kind": f"{peak_kind} hbm_gbs (copy)",
                "algorithmic_bytes_per_launch": io_bytes,
                "tensor_tflops": flops / kernel_s / 1e12, "tensor_peak_tflops": tpk}

    cpu = None
    if not args.no_cpu_baseline and world == 1 and not noncausal:
        cores = host_cores()
        heads = sample_heads(w, cores)
        sub = {kk: (vv[heads] if kk in ("q", "k", "v", "lam") and vv is not None else vv)
               for kk, vv in inp.items()}
        val, dt = cpu_baseline(w, sub, len(heads), cores)
        cpu = {"value": val, "unit": "tokens/s", "cores": min(cores, len(heads)),
               "kind": "oracle",
               "sample": f"{len(heads)} of {B * H} heads x L={L}, chunk-size-1 recurrence in "
                         f"fp64, {dt:.1f} s wall",
               "one_core": cpu_baseline_one_core(w, sub)}

    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if w["dtype"] == "bf16" else "f32", "data": "synthetic",
            "config": dict(workload_config(args.workload, w, C),
                           l2="inputs larger than L2" if flush is None else
                           "L2 flushed between steps (2x L2 buffer written)",
                           path={1: "simt", 2: "tc"}.get(plan["path"], plan["path"]),
                           op=args.op,
                           parallelism=f"heads independent; weak scaling over {world} GPU(s)"),
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "clocks": clk,
            "gpu_launches": plan["n_launches"] * args.steps}
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


def run_decode(args):
    """Decoding steps: each timed step is one la_decode_step over every (b, h) head of the
    workload (one token per head).  A step streams the fp32 state through the SMs once, so
    the roofline is HBM: bytes = state (and normaliser) read + written + q, k, v, out (+ the
    token's level weights).  L2 is flushed between steps when the state fits in it."""
    import torch

    import chunkwise_causal_linear_gb300 as la
    from chunkwise_causal_linear_gb300 import build as la_build
    if not la_build.up_to_date():
        la_build.build()
    torch.cuda.set_device(0)
    w = dict(synth.WORKLOADS[args.workload])
    if args.B:
        w["B"] = args.B
    if args.H:
        w["H"] = args.H
    B, H, dk, dv = w["B"], w["H"], w["dk"], w["dv"]
    T = args.warmup + args.steps
    wt = dict(w, L=T)
    inp = synth.make_inputs(wt, args.seed)
    es = 2 if w["dtype"] == "bf16" else 4

    def dev(x, d):
        if w["dtype"] == "bf16":
            t = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16)
        else:
            t = torch.from_numpy(x)
        return t.reshape(B, H, T, d).cuda()

    q, k, v = dev(inp["q"], dk), dev(inp["k"], dk), dev(inp["v"], dv)
    toks = [(q[:, :, t].contiguous(), k[:, :, t].contiguous(), v[:, :, t].contiguous()) for t in range(T)]
    omega = None if inp["omega"] is None else torch.from_numpy(inp["omega"]).cuda()
    lams = None
    nl = 0
    if inp["lam"] is not None:
        # levels for positions up to T (one more than a forward over T rows uses)
        nl = synth.num_levels(T + 1) + 1
        lam = np.zeros((B, H, T, nl), dtype=np.float32)
        src = inp["lam"].reshape(B, H, T, -1)
        lam[..., :src.shape[-1]] = src
        lam_d = torch.from_numpy(lam).cuda()
        lams = [lam_d[:, :, t].contiguous() for t in range(T)]
    D = w["m"] if w["fm"] == "favor" else dk
    S, z = la.decode_state(B, H, dk, dv, w["fm"], w["m"], nl, w["normalize"])
    out = torch.empty((B, H, dv), dtype=q.dtype, device="cuda")
    state_bytes = S.numel() * 4 + (z.numel() * 4 if z is not None else 0)
    flush = None
    if state_bytes < 2 * L2_BYTES:
        flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def step(t):
        la.decode_step(*toks[t], S, z, t=t, feature_map=w["fm"], omega=omega,
                       normalize=w["normalize"], level_weights=lams[t] if lams else None, out=out,
                       stream=stream.cuda_stream)

    def algo_bytes(t):
        per_level = B * H * D * (dv + (1 if w["normalize"] else 0)) * 4
        lv = (nl - 1) if nl else 1
        if nl:
            x, r = t + 1, 0
            while not (x >> r) & 1:
                r += 1
            written = r + 1
        else:
            written = 1
        return (lv + written) * per_level + B * H * ((2 * dk + 2 * dv) * es + nl * 4)

    for t in range(args.warmup):
        step(t)
    torch.cuda.synchronize()
    st = la.la_last_device_status(stream.cuda_stream)
    if st != la.LA_OK:
        raise la.LAError(st, "device status after warm-up")
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for i in range(args.steps):
        if flush is not None:
            flush.zero_()
        evs[i][0].record(stream)
        step(args.warmup + i)
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    times = [a.elapsed_time(b) for a, b in evs]
    t_ms = sum(times)
    ms = t_ms / args.steps
    byts = sum(algo_bytes(args.warmup + i) for i in range(args.steps)) / args.steps
    peaks, peak_kind = measured_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    achieved = byts / (ms / 1e3) / 1e9
    line = {"metric": "decode tokens/sec (B·H tokens per la_decode_step)", "op": "decode",
            "value": B * H * args.steps / (t_ms / 1e3), "unit": "tokens/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if w["dtype"] == "bf16" else "f32", "data": "synthetic",
            "config": {"workload": args.workload, "B": B, "H": H, "dk": dk, "dv": dv,
                       "feature_map": w["fm"], "m": w["m"], "normalize": bool(w["normalize"]),
                       "num_levels": nl, "state_bytes": state_bytes,
                       "l2": "L2 flushed between steps (2x L2 buffer written)" if flush is not None
                       else "state larger than L2"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                         "frac": achieved / hbm, "traffic": None,
                         "peak_kind": f"{peak_kind} hbm_gbs (copy)",
                         "algorithmic_bytes_per_launch": byts},
            "cpu_baseline": None, "e2e": None, "clocks": clk, "gpu_launches": args.steps}
    print(json.dumps(line), flush=True)
    return 0


def run_backward(args):
    """Backward passes: each timed step is one la_chunked_bwd (la_chunked_bwd_ll for the
    log-linear mask) over the whole workload.  Algorithmic bytes per step: q, k, v, dout (and
    the level weights) read and dq, dk, dv written once each."""
    import torch

    import chunkwise_causal_linear_gb300 as la
    from chunkwise_causal_linear_gb300 import build as la_build
    if not la_build.up_to_date():
        la_build.build()
    torch.cuda.set_device(0)
    w = dict(synth.WORKLOADS[args.workload])
    for key in ("B", "H", "L"):
        if getattr(args, key):
            w[key] = getattr(args, key)
    ll = bool(w.get("loglinear"))
    B, H, L, dk, dv = w["B"], w["H"], w["L"], w["dk"], w["dv"]
    C = args.C if args.C is not None else w["C"]
    gamma = w.get("gamma") or 1.0
    inp = synth.make_inputs(w, args.seed)
    do_bits = synth.tensor_values(args.seed, synth.T_DOUT, B, H, L, dv, "normal", 1.0, w["dtype"])
    es = 2 if w["dtype"] == "bf16" else 4

    def dev(x, d):
        if w["dtype"] == "bf16":
            t = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16)
        else:
            t = torch.from_numpy(x)
        return t.reshape(B, H, L, d).cuda()

    q, k, v, do = dev(inp["q"], dk), dev(inp["k"], dk), dev(inp["v"], dv), dev(do_bits, dv)
    omega = None if inp["omega"] is None else torch.from_numpy(inp["omega"]).cuda()
    fm = la.make_feature_map(w["fm"], w["m"], omega.data_ptr() if omega is not None else 0)
    dtype = la.LA_BF16 if w["dtype"] == "bf16" else la.LA_F32
    lam = None if inp["lam"] is None else torch.from_numpy(inp["lam"]).reshape(B, H, L, -1).cuda()
    nl = 0 if lam is None else lam.shape[-1]
    if ll:
        need = la.la_chunked_bwd_ll_workspace_bytes(B, H, L, dk, dv, C, fm, int(w["normalize"]), nl,
                                                    dtype)
    else:
        need = la.la_chunked_bwd_workspace_bytes(B, H, L, dk, dv, C, fm, int(w["normalize"]), dtype)
    if need == 0:
        raise SystemExit("--op backward: unsupported sizes")
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    dq, dk_t, dv_t = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    stream = torch.cuda.current_stream()

    def step():
        if ll:
            r = la.la_chunked_bwd_ll(q.data_ptr(), k.data_ptr(), v.data_ptr(), do.data_ptr(),
                                     dq.data_ptr(), dk_t.data_ptr(), dv_t.data_ptr(), B, H, L, dk,
                                     dv, C, fm, int(w["normalize"]), lam.data_ptr(), nl, dtype,
                                     ws.data_ptr(), need, stream.cuda_stream)
        else:
            r = la.la_chunked_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), do.data_ptr(),
                                  dq.data_ptr(), dk_t.data_ptr(), dv_t.data_ptr(), B, H,
                                  L, dk, dv, C, fm, int(w["normalize"]), float(gamma), dtype,
                                  ws.data_ptr(), need, stream.cuda_stream)
        if r != la.LA_OK:
            raise la.LAError(r, "la_chunked_bwd_ll" if ll else "la_chunked_bwd")

    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize()
    st = la.la_last_device_status(stream.cuda_stream)
    if st != la.LA_OK:
        raise la.LAError(st, "device status after warm-up")
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for i in range(args.steps):
        evs[i][0].record(stream)
        step()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    t_ms = sum(a.elapsed_time(b) for a, b in evs)
    ms = t_ms / args.steps
    byts = B * H * L * (es * (4 * dk + 3 * dv) + 4 * nl)
    peaks, peak_kind = measured_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    achieved = byts / (ms / 1e3) / 1e9
    # Launches per step.  Tensor-core routes: every pass is one launch, or two where the plan
    # splits the sequence (a totals launch first), as for a forward of the same B, H, L.
    # Identity / elu+1 (dk = dv in {64, 128}; the decay without the normaliser): 3 passes
    # (+ Z, num, suffix and a prep kernel with the normaliser), elu+1's feature kernel, and a
    # chain kernel for elu+1 or the normaliser.  FAVOR+ (dk = dv = 64, m = 128, 256 or 512):
    # 2 feature kernels, 3 passes per 128-feature half (+ 3 and a prep kernel with the
    # normaliser), 1 chain kernel.  The generic route: 2 features, v', prep, 3 passes, 2
    # chain, 1 cast (+ 1 pass).
    nz = bool(w["normalize"])
    favor_tc = (w["dtype"] == "bf16" and w["fm"] == "favor" and gamma == 1.0 and L >= 128
                and dk == dv == 64 and w["m"] in (128, 256, 512) and not ll)
    tc_route = favor_tc or (w["dtype"] == "bf16" and w["fm"] in ("identity", "elu1")
                            and (gamma == 1.0 or (gamma >= 0.5 and not nz))
                            and L >= 128 and dk == dv and dk in (64, 128) and not ll)
    if tc_route:
        _, pplan = la.la_chunked_plan(B, H, L, 64, 64, 64, la.make_feature_map("identity"), 0, 0, 0,
                                      dtype, la.LA_PATH_TC, 0)
        per_pass = pplan["n_launches"]
        if favor_tc:
            nh = w["m"] // 128
            launches = 3 + (1 if nz else 0) + per_pass * nh * (6 if nz else 3)
        else:
            launches = per_pass * (6 if nz else 3) + (1 if nz else 0)
            launches += (1 if w["fm"] == "elu1" else 0) + (1 if (nz or w["fm"] == "elu1") else 0)
    else:
        launches = 10 + (1 if nz else 0)
    if ll:  # two anti-causal sums of two launches each instead of one pass each
        launches += 2
    line = {"metric": "backward tokens/sec (B·H·L/s, %s)" % ("la_chunked_bwd_ll" if ll else "la_chunked_bwd"),
            "op": "backward",
            "value": B * H * L * args.steps / (t_ms / 1e3), "unit": "tokens/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if w["dtype"] == "bf16" else "f32", "data": "synthetic",
            "config": dict(workload_config(args.workload, w, C), path="tc" if tc_route else "simt",
                           l2="inputs larger than L2"),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                         "frac": achieved / hbm, "traffic": None,
                         "peak_kind": f"{peak_kind} hbm_gbs (copy)",
                         "algorithmic_bytes_per_launch": byts},
            "cpu_baseline": None, "e2e": None, "clocks": clk,
            "gpu_launches": launches * args.steps}
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    if args.op == "decode":
        return run_decode(args)
    if args.op == "backward":
        return run_backward(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
