"""Benchmark of the Dobb optimizer step on the GPT-2 XL parameter set, B = 16.

Workload: 48 layers x {q, k, v, o: 1600 x 1600; fc: 6400 x 1600; proj:
1600 x 6400} plus the tied 50257 x 1600 token embedding (289 matrices,
1,554,971,200 parameters), bf16 parameters and gradients, fp32 momentum,
B = 16 (k = 100 for n = 1600, k = 400 for n = 6400), 8 x 1024 bf16 activation
tokens per matrix with effective rank varying 10% -> 40% over depth, basis
refresh every 10 steps.  A step is one pass of the hot path: accumulate the
block moments, refresh the bases when t % 10 == 0, update every matrix.

value = parameters updated per second (whole job); ms_per_step is the mean
over the timed steps, which contain refresh steps at the configured period.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "Dobb optimizer step ms (GPT-2 XL, B=16) and params/s; % of roofline"
UNIT = "params/s"
B_BLOCKS = 16
REFRESH = 10
N_TOKENS = 8192
BETA1, BETA2, LR, SCALE = 0.95, 0.99, 0.02, 1.0


def _env_rank():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


# ---------------------------------------------------------------------------
# algorithmic work per launch (units: bytes / flops), see the design notes
# ---------------------------------------------------------------------------

def work_model(shapes, B, N, pbytes=2, xbytes=2, refresh="eigh", orth_steps=1, norm="sign",
               sides=None):
    upd_bytes = upd_flops = acc_bytes = acc_flops = ref_flops = ref_bytes = 0
    for i, (m, n) in enumerate(shapes):
        if sides is not None and sides[i] == "output":
            m, n = n, m   # Dobb-G: the same work on the transposed problem
        k = n // B
        # update: G read, M read + write, W read + write, Q_b read once
        upd_bytes += m * n * (pbytes + 4 + 4 + 2 * pbytes) + 4 * B * k * k
        if norm == "l2":
            # the column norms run over all rows before any row is updated: the
            # momentum is read a second time
            upd_bytes += 4 * m * n
        upd_flops += 4 * k * m * n
        # accumulate: X read, A read + write (symmetric: N k (k+1) flops)
        acc_bytes += xbytes * N * n + 8 * B * k * k
        acc_flops += B * N * k * (k + 1)
        # refresh: 9 k^3 flops per block (symmetric eigendecomposition with
        # vectors), or per orthogonal-iteration step 2 k^3 (A Q) + k^3 (Gram,
        # symmetric) + k^3 / 3 (Cholesky) + k^3 (triangular solve); A read,
        # Q and Lambda written
        ref_flops += B * k ** 3 * (9 if refresh == "eigh" else orth_steps * 13 / 3)
        ref_bytes += 8 * B * k * k + 4 * B * k
    return dict(update_bytes=upd_bytes, update_flops=upd_flops, acc_bytes=acc_bytes,
                acc_flops=acc_flops, refresh_flops=ref_flops, refresh_bytes=ref_bytes)


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid=None):
        self.uuid = uuid
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for l in self.lines:
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 10:
                continue
            if self.uuid and self.uuid not in parts[1]:
                continue
            rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = sorted(float(r[2]) for r in rows if r[2].replace(".", "").isdigit())
        mx = max(float(r[3]) for r in rows if r[3].replace(".", "").isdigit())
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for nm, v in zip(names, r[6:10]):
                if v.strip().lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(rows)}


# ---------------------------------------------------------------------------
# synthetic inputs on the device (seeded)
# ---------------------------------------------------------------------------

def make_inputs(torch, shapes, layers, device, seed, n_xsets=2, sides=None):
    """X_i (N x n, bf16) per matrix with layer-dependent effective rank,
    G_i = D X_i / N (bf16), W_i ~ N(0, 0.02^2) (bf16).  For an output-side
    (Dobb-G) matrix X_i are output gradients (N x m) of the same recipe and
    G_i = X_i^T D / N.  Generated on the device with torch's seeded
    generator; the spectra come from the shared input module."""
    from block_eigenbasis_preconditioning_gb300 import inputs as I
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    import numpy as np
    nl = max(layers) if layers else 1
    lam_cache = {}
    haar_cache = {}
    Xsets = [[] for _ in range(n_xsets)]
    Gs, Ws = [], []
    for i, ((m, n), li) in enumerate(zip(shapes, layers)):
        out = sides is not None and sides[i] == "output"
        if out:
            m, n = n, m   # X spans the output axis; G is built transposed below
        eff = I.layer_rank_schedule(min(li, nl - 1), nl) if li < nl else 0.10
        key = (n, round(eff, 6))
        if key not in lam_cache:
            lam = I.geometric_spectrum(n, eff)
            lam = lam * (n / lam.sum())
            lam_cache[key] = torch.tensor(lam, dtype=torch.float32, device=device).sqrt_()
        sq = lam_cache[key]
        if n not in haar_cache:
            haar_cache[n] = torch.tensor(I.haar_orthogonal(n, np.random.default_rng(seed + n)),
                                         dtype=torch.float32, device=device)
        # per-matrix eigenvectors: the shared Haar basis with permuted, sign-flipped rows
        perm = torch.randperm(n, generator=g, device=device)
        flip = torch.randint(0, 2, (n, 1), generator=g, device=device).float() * 2 - 1
        q = haar_cache[n][perm] * flip
        for s in range(n_xsets):
            Z = torch.randn(N_TOKENS, n, generator=g, device=device)
            X = (Z * sq.unsqueeze(0)) @ q.T
            Xsets[s].append(X.to(torch.bfloat16))
            del Z, X
        D = torch.randn(m, N_TOKENS, generator=g, device=device)
        G = (D @ Xsets[0][-1].float()) / N_TOKENS
        Gs.append((G.T if out else G).contiguous().to(torch.bfloat16))
        del D, G
        W = torch.randn(m, n, generator=g, device=device) * 0.02
        Ws.append((W.T if out else W).contiguous().to(torch.bfloat16))
    return Xsets, Gs, Ws


def flush_l2(torch, buf):
    buf.zero_()


def _kernel_source_sha(name):
    p = os.path.join(ROOT, "block_eigenbasis_preconditioning_gb300", "csrc", name)
    try:
        with open(p, "rb") as f:
            return hashlib.sha256(f.read()).hexdigest()[:16]
    except OSError:
        return None


def _traffic_for(kernel_key):
    """dram bytes of that kernel per step (all its launches in one step) from a
    committed ncu summary, if it was taken on the current source of the kernel."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)
        e = t.get(kernel_key)
        if e and e.get("source_sha") == _kernel_source_sha(e.get("source")):
            return e.get("bytes_per_step")
    except Exception:
        pass
    return None


# ---------------------------------------------------------------------------
# CPU baseline: the oracle on a bounded sample
# ---------------------------------------------------------------------------

def cpu_baseline(layers_sample=2, seed=0, basis="f32", refresh="eigh", orth_steps=1, norm="sign",
                 side="input"):
    import numpy as np
    from block_eigenbasis_preconditioning_gb300 import inputs as I
    from oracle import dobb as O
    rng = np.random.default_rng(seed)
    shapes = []
    for _ in range(layers_sample):
        shapes += [(1600, 1600)] * 4 + [(6400, 1600), (1600, 6400)]
    params = sum(m * n for m, n in shapes)
    orc = O.DobbOracle(shapes, B_BLOCKS, BETA1, BETA2, refresh_period=0, scale_s=SCALE,
                       param_dtype="bf16", eig_method="lapack", basis_dtype=basis,
                       refresh_method=refresh, orth_steps=orth_steps, norm=norm, side=side)
    Xs = [I.round_bf16_np(rng.standard_normal((N_TOKENS, m if side == "output" else n))
                          .astype(np.float32)) for m, n in shapes]
    Gs = [I.round_bf16_np((rng.standard_normal((m, n)) * 1e-3).astype(np.float32)) for m, n in shapes]
    Ws = [I.round_bf16_np((rng.standard_normal((m, n)) * 0.02).astype(np.float32)) for m, n in shapes]
    t0 = time.perf_counter()
    orc.accumulate(Xs)
    t1 = time.perf_counter()
    orc.refresh()
    t2 = time.perf_counter()
    orc.step(Ws, Gs, LR)
    t3 = time.perf_counter()
    acc, ref, upd = t1 - t0, t2 - t1, t3 - t2
    step_s = acc + upd + ref / REFRESH
    return {"value": params / step_s, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{layers_sample} GPT-2 XL layers ({params} params, 12 matrices), one "
                      f"accumulate (N={N_TOKENS}) + one "
                      f"{'LAPACK' if refresh == 'eigh' else 'orthogonal-iteration'} refresh + one "
                      f"update in fp64 numpy; "
                      f"amortized as accumulate + update + refresh/{REFRESH}",
            "seconds": {"accumulate": acc, "refresh": ref, "update": upd}}


def workload_config(args, n_matrices=None, params=None):
    """The workload both arms report (the reference arm runs a bounded sample
    of it on the host, described in its cpu_baseline)."""
    if args.layers is None:
        name = ("gpt2-xl B=16: 289 matrices, 1.555e9 params, bf16 W/G, fp32 M, "
                "X 8192 bf16 tokens/matrix, refresh every 10")
    else:
        name = (f"gpt2-xl shapes, first {args.layers} layers ({n_matrices} matrices, "
                f"{params} params), B=16")
    return {"workload": name, "B": B_BLOCKS, "refresh_period": REFRESH, "tokens": N_TOKENS,
            "basis": args.basis, "norm": args.norm, "side": args.side,
            "refresh": args.refresh if args.refresh == "eigh" else f"orth x{args.orth_steps}",
            "l2": "inputs larger than L2 (22 GB streamed per step)",
            "parallelism": "single GPU"}


def run_reference(args):
    rank, world, _ = _env_rank()
    if rank != 0:
        return 0
    steps = []
    res = None
    for _ in range(max(1, args.steps)):
        res = cpu_baseline(layers_sample=1, basis=args.basis, refresh=args.refresh,
                           orth_steps=args.orth_steps, norm=args.norm, side=args.side)
        steps.append(res["value"])
    v = sorted(steps)[len(steps) // 2]
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": 0, "ms_per_step": 1.5549712e9 / v * 1e3 if v else None,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(args),
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": res["cores"], "kind": "oracle",
                             "sample": res["sample"]},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def run_gpu(args):
    import torch
    import torch.distributed as dist
    from block_eigenbasis_preconditioning_gb300 import Dobb
    from block_eigenbasis_preconditioning_gb300 import inputs as I

    rank, world, local = _env_rank()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    ms = I.gpt2_xl_shapes(include_embedding=args.layers is None)
    shapes, layers = ms.shapes, ms.layer
    if args.layers is not None:
        keep = [i for i, li in enumerate(layers) if li < args.layers]
        shapes = [shapes[i] for i in keep]
        layers = [layers[i] for i in keep]
    params = sum(m * n for m, n in shapes)
    # Dobb-G blocks the output axis of every layer matrix; the token
    # embedding (50257 rows: no 16 equal blocks) stays on the input side
    sides = [("output" if args.side == "output" and m % B_BLOCKS == 0 and m // B_BLOCKS <= 1024
              else "input") for m, n in shapes]
    Xsets, Gs, Ws = make_inputs(torch, shapes, layers, device, seed=1234 + rank, sides=sides)
    opt = Dobb(shapes, B_BLOCKS, BETA1, BETA2, refresh_period=REFRESH, scale_s=SCALE,
               param_dtype="bf16", act_dtype="bf16", device=device, basis_dtype=args.basis,
               refresh=args.refresh, orth_steps=args.orth_steps, norm=args.norm, side=sides)
    stream = torch.cuda.current_stream()
    moments = opt.tensor("moments")

    def one_step(t, xs, ev=None):
        if ev is not None:
            ev[0].record(stream)
        opt.accumulate(xs)
        if ev is not None:
            ev[1].record(stream)
        if world > 1 and t % REFRESH == 0:
            dist.all_reduce(moments, op=dist.ReduceOp.SUM)
            moments.div_(world)
        if ev is not None:
            ev[2].record(stream)
        opt.step(Ws, Gs, LR)
        if ev is not None:
            ev[3].record(stream)

    for t in range(args.warmup):
        one_step(opt.t, Xsets[t % len(Xsets)])
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()

    # timed region
    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    is_refresh = []
    clocks = ClockSampler(getattr(torch.cuda.get_device_properties(device), "uuid", None) and
                          str(torch.cuda.get_device_properties(device).uuid))
    clocks.start()
    launches0 = opt.launch_count
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(K):
        t = opt.t
        is_refresh.append(t % REFRESH == 0)
        one_step(t, Xsets[t % len(Xsets)], evs[i])
    end.record(stream)
    torch.cuda.synchronize()
    launches = opt.launch_count - launches0
    ms_total = start.elapsed_time(end)
    clk = clocks.stop()
    if world > 1:
        tt = torch.tensor([ms_total], device=device)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        ms_total = float(tt.item())
        dist.barrier()
    ms_step = ms_total / K
    acc_ms = [evs[i][0].elapsed_time(evs[i][1]) for i in range(K)]
    upd_ref_ms = [evs[i][2].elapsed_time(evs[i][3]) for i in range(K)]
    upd_ms = [v for v, r in zip(upd_ref_ms, is_refresh) if not r]
    ref_steps = [v for v, r in zip(upd_ref_ms, is_refresh) if r]
    mean = lambda v: sum(v) / len(v) if v else None
    upd_mean = mean(upd_ms)
    refresh_ms = (mean(ref_steps) - upd_mean) if (ref_steps and upd_mean is not None) else None

    # refresh measured on its own when the timed window held none
    if refresh_ms is None:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        opt.refresh()
        e1.record(stream)
        torch.cuda.synchronize()
        refresh_ms = e0.elapsed_time(e1)

    hbm, bf16, peak_kind = _peaks()
    wm = work_model(shapes, B_BLOCKS, N_TOKENS, refresh=args.refresh, orth_steps=args.orth_steps,
                    norm=args.norm, sides=sides)
    ffma_update = args.norm != "sign"
    alu_peak_tflops = 152 * 128 * 2 * 2.07e9 / 1e12  # FP32 lanes x FMA x max SM clock
    phases = {
        "update": {"ms": upd_mean, "kernel": "step_ffma_kernel" if ffma_update else "step_tc_kernel",
                   "bound": "hbm",
                   "achieved": wm["update_bytes"] / (upd_mean * 1e-3) / 1e9 if upd_mean else None,
                   "peak": hbm, "unit": "GB/s", "flops": wm["update_flops"], "bytes": wm["update_bytes"]},
        "accumulate": {"ms": mean(acc_ms), "kernel": "syrk_tc_kernel", "bound": "hbm",
                       "achieved": wm["acc_bytes"] / (mean(acc_ms) * 1e-3) / 1e9,
                       "peak": hbm, "unit": "GB/s", "flops": wm["acc_flops"], "bytes": wm["acc_bytes"]},
        "refresh": {"ms": refresh_ms, "kernel": "jacobi_kernel" if args.refresh == "eigh" else "orth_kernel",
                    "bound": "alu",
                    "achieved": wm["refresh_flops"] / (refresh_ms * 1e-3) / 1e12,
                    "peak": alu_peak_tflops, "unit": "TFLOP/s", "flops": wm["refresh_flops"]},
    }
    for p in phases.values():
        p["frac"] = p["achieved"] / p["peak"] if p.get("achieved") else None
    # dominant kernel: most device time per refresh cycle
    share = {"update": (upd_mean or 0) * (REFRESH - 0), "accumulate": mean(acc_ms) * REFRESH,
             "refresh": refresh_ms}
    dom = max(share, key=share.get)
    d = phases[dom]
    roofline = {"bound": d["bound"], "achieved": d["achieved"], "peak": d["peak"], "unit": d["unit"],
                "frac": d["frac"], "traffic": _traffic_for(d["kernel"]), "kernel": d["kernel"],
                "peak_source": peak_kind}

    # end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(torch, opt, Xsets[0], Gs, Ws, K, stream, params, world)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        try:
            cpu = cpu_baseline(basis=args.basis, refresh=args.refresh, orth_steps=args.orth_steps,
                               norm=args.norm, side=args.side)
        except Exception as ex:  # pragma: no cover
            cpu = {"error": repr(ex)}

    if rank == 0:
        amort = mean(acc_ms) + upd_mean + refresh_ms / REFRESH if upd_mean else None
        line = {"metric": METRIC, "value": params * world / (ms_step * 1e-3), "unit": UNIT,
                "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": ms_step,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
                "data": "synthetic",
                "config": dict(workload_config(args, len(shapes), params),
                               refresh_steps_timed=sum(is_refresh),
                               parallelism=f"dp{world} replicas" if world > 1 else "single GPU"),
                "phases_ms": {"accumulate": mean(acc_ms), "update": upd_mean, "refresh": refresh_ms,
                              "amortized_step": amort},
                "phases": phases, "roofline": roofline, "clocks": clk,
                "gpu_launches": launches, "e2e": e2e, "cpu_baseline": cpu}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def _bind_to_gpu_local_cpus(torch):
    """Run this process on the host cores attached to the current GPU while the
    pinned input buffers are allocated, so that their pages land in that
    socket's memory (host buffers on the other socket cross the CPU-CPU link
    on every copy).  Best effort: a system that does not expose the GPU's
    local CPUs is left as is."""
    try:
        props = torch.cuda.get_device_properties(torch.cuda.current_device())
        bus = "%04x:%02x:%02x.0" % (props.pci_domain_id, props.pci_bus_id, props.pci_device_id)
        with open(f"/sys/bus/pci/devices/{bus}/local_cpulist") as f:
            spec = f.read().strip()
        cpus = set()
        for part in spec.split(","):
            lo, _, hi = part.partition("-")
            cpus.update(range(int(lo), int(hi or lo) + 1))
        if cpus:
            os.sched_setaffinity(0, cpus)
    except Exception:
        pass


def run_e2e(torch, opt, X, G, W, K, stream, params, world):
    """Each step copies that step's activations and gradients from pinned
    host memory, runs accumulate (+ refresh) + step through the public API,
    and reads the per-block update norms back to the host.  The copies of
    step i+1 run on two copy streams into a second set of device buffers
    while step i computes (double buffering); a step's compute waits for its
    own inputs, and a buffer set is refilled only after the step that read it."""
    prev_cpus = os.sched_getaffinity(0)
    _bind_to_gpu_local_cpus(torch)
    Xh = [x.cpu().pin_memory() for x in X]
    Gh = [g.cpu().pin_memory() for g in G]
    os.sched_setaffinity(0, prev_cpus)   # the pages are placed; the rest may use every core
    Xd = [[torch.empty_like(x) for x in X] for _ in range(2)]
    Gd = [[torch.empty_like(g) for g in G] for _ in range(2)]
    h2d = sum(x.numel() * x.element_size() for x in Xh) + sum(g.numel() * g.element_size() for g in Gh)
    stats = torch.empty(opt.num_blocks * 4, dtype=torch.float32).pin_memory()
    d2h = stats.numel() * 4
    st_dev = opt.tensor("stats")
    cx, cg = torch.cuda.Stream(), torch.cuda.Stream()
    copied = [torch.cuda.Event() for _ in range(2)]
    consumed = [torch.cuda.Event() for _ in range(2)]

    def issue_copies(i):
        b = i % 2
        for cs, dst, src in ((cx, Xd[b], Xh), (cg, Gd[b], Gh)):
            if i >= 2:
                cs.wait_event(consumed[b])   # step i-2 has read this buffer set
            with torch.cuda.stream(cs):
                for d, h in zip(dst, src):
                    d.copy_(h, non_blocking=True)
        ev_g = torch.cuda.Event()
        ev_g.record(cg)
        copied[b].record(cx)
        return ev_g

    torch.cuda.synchronize()
    t0 = time.perf_counter()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    cx.wait_stream(stream)
    cg.wait_stream(stream)
    pending = issue_copies(0)
    for i in range(K):
        b = i % 2
        stream.wait_event(copied[b])
        stream.wait_event(pending)
        nxt = issue_copies(i + 1) if i + 1 < K else None
        opt.accumulate(Xd[b])
        opt.step(W, Gd[b], LR)
        consumed[b].record(stream)
        stats.copy_(st_dev, non_blocking=True)
        pending = nxt
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / K
    return {"value": params * world / (ms * 1e-3), "unit": UNIT, "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "wall_ms_per_step": (time.perf_counter() - t0) * 1e3 / K,
            "overlap": "inputs of step i+1 copied on two streams during step i"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--refresh", default="eigh", choices=["eigh", "orth"],
                    help="eigh: complete eigendecomposition; orth: orthogonal iteration with "
                         "Cholesky QR (the pages' principal refresh)")
    ap.add_argument("--orth-steps", type=int, default=1)
    ap.add_argument("--norm", default="sign", choices=["sign", "l2"],
                    help="coefficient normalisation: sign (Dobb) or l2 (Dobb-l2, FP32 kernels)")
    ap.add_argument("--side", default="input", choices=["input", "output"],
                    help="input: Dobb (blocks of the input axis, activation moments); output: "
                         "Dobb-G (blocks of the output axis, output-gradient moments)")
    ap.add_argument("--basis", default="f32", choices=["f32", "bf16"],
                    help="precision of the basis the update multiplies with (bf16: the "
                         "pages' principal storage setting)")
    ap.add_argument("--layers", type=int, default=None,
                    help="smaller model of the same layer shapes (first L layers, no "
                         "embedding), for profiler captures")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
