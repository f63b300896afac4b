"""Benchmark of the Dobb optimizer step.

Default workload (the headline): the GPT-2 XL parameter set, B = 16 -- 48
layers x {q, k, v, o: 1600 x 1600; fc: 6400 x 1600; proj: 1600 x 6400} plus
the tied 50257 x 1600 token embedding (289 matrices, 1,554,971,200
parameters), bf16 parameters and gradients, fp32 momentum, k = 100 for
n = 1600 and k = 400 for n = 6400, 8 x 1024 bf16 activation tokens per
matrix with effective rank varying 10 % -> 40 % over depth, refresh every
10 steps.  A step is one pass of the hot path: accumulate the block moments,
refresh the bases when t % T == 0, update every matrix.  Inputs drift: each
step takes the next of a pool of independently drawn activation / gradient
sets resident in HBM.

Other workloads (--config): gpt2-small (72 fp32 matrices, B = 16, 4096
tokens, refresh every 10), single (one fp32 768 x 768 matrix, B = 4, refresh
every 5), llama3-8b (226 bf16 matrices, B = 32, 4096 tokens, refresh every
20), stress-b16 / stress-b4 / stress-b1 (GPT-2 XL shapes, every block
re-eigensolved at every step from fresh SPD blocks with relative gaps
>= 1e-3 and condition number 1e6).

value = parameters updated per second over the whole job; ms_per_step is the
mean over the timed steps, which contain refresh steps at the configured
period.

  python bench.py [--config NAME] [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
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

CONFIGS = {
    "gpt2-xl": dict(model="gpt2-xl", B=16, T=10, N=8192, pdt="bf16", adt="bf16", eff="layers",
                    pool=10, kind="train"),
    "gpt2-small": dict(model="gpt2-small", B=16, T=10, N=4096, pdt="f32", adt="f32", eff=0.20,
                       pool=10, kind="train"),
    "single": dict(model="single", B=4, T=5, N=1024, pdt="f32", adt="f32", eff=0.15, pool=10,
                   kind="train"),
    "llama3-8b": dict(model="llama3-8b", B=32, T=20, N=4096, pdt="bf16", adt="bf16", eff=0.15,
                      pool=3, kind="train"),
    "stress-b16": dict(model="gpt2-xl", B=16, T=1, N=0, pdt="bf16", adt="bf16", pool=2,
                       kind="stress"),
    "stress-b4": dict(model="gpt2-xl", B=4, T=1, N=0, pdt="bf16", adt="bf16", pool=2,
                      kind="stress"),
    "stress-b1": dict(model="gpt2-xl", B=1, T=1, N=0, pdt="bf16", adt="bf16", pool=2,
                      kind="stress"),
}
BETA1, BETA2, LR, SCALE = 0.95, 0.99, 0.02, 1.0


def _env_rank():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def _measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "MEASURED_PEAKS.json (copy bandwidth, cuBLAS bf16)"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


def model_shapes(name, layers=None):
    from block_eigenbasis_preconditioning_gb300 import inputs as I
    ms = {"gpt2-xl": lambda: I.gpt2_xl_shapes(include_embedding=layers is None),
          "gpt2-small": I.gpt2_small_shapes, "llama3-8b": I.llama3_8b_shapes,
          "single": I.single_matrix_shapes}[name]()
    shapes, lay = list(ms.shapes), list(ms.layer)
    if layers is not None:
        keep = [i for i, li in enumerate(lay) if li < layers]
        shapes = [shapes[i] for i in keep]
        lay = [lay[i] for i in keep]
    return shapes, lay


# ---------------------------------------------------------------------------
# algorithmic work per step (bytes / flops); see the design notes
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
            upd_bytes += 4 * m * n   # the column norms read the momentum a second time
        upd_flops += 4 * k * m * n
        # accumulate: X read, A read + write (symmetric: N k (k+1) flops)
        acc_bytes += xbytes * N * n + 8 * B * k * k
        acc_flops += B * N * k * (k + 1)
        # refresh: 9 k^3 flops per block (symmetric eigendecomposition with
        # vectors), or per orthogonal-iteration step 2 k^3 (A Q) + k^3 (Gram,
        # symmetric) + k^3 / 3 (Cholesky) + k^3 (triangular solve); A read, Q
        # and Lambda written
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
# throughput probes and host link rates
# ---------------------------------------------------------------------------

def probe_peaks(torch):
    """Roofline denominators measured in this process with the library's
    throughput probes (best of three launches each): FP32 FFMA, TF32 and
    BF16 tcgen05, TF32 mma.sync."""
    from block_eigenbasis_preconditioning_gb300 import binding
    buf = torch.empty(16 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    out = {}
    for which, iters in (("ffma", 20000), ("tc_tf32", 20000), ("tc_bf16", 20000),
                         ("mma_sync_tf32", 20000)):
        binding.peak_probe(which, buf.data_ptr(), buf.numel(), iters // 20, stream)
        best = 0.0
        for _ in range(3):
            ms, fl = binding.peak_probe(which, buf.data_ptr(), buf.numel(), iters, stream)
            best = max(best, fl / (ms * 1e-3) / 1e12)
        out[which + "_tflops"] = best
    out["source"] = "in-process probes (dobb_peak_probe), best of 3"
    del buf
    return out


def host_link_rates(torch, nbytes=1 << 30):
    """Pinned host <-> device copy rates (GB/s, best of 3)."""
    h = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    res = {}
    for name, fn in (("h2d_gbs", lambda: d.copy_(h, non_blocking=True)),
                     ("d2h_gbs", lambda: h.copy_(d, non_blocking=True))):
        best = 0.0
        for _ in range(3):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            best = max(best, nbytes / (e0.elapsed_time(e1) * 1e-3) / 1e9)
        res[name] = best
    del h, d
    return res


# ---------------------------------------------------------------------------
# synthetic inputs on the device (seeded)
# ---------------------------------------------------------------------------

def _eff_for(cfg, lay):
    from block_eigenbasis_preconditioning_gb300 import inputs as I
    if cfg["eff"] != "layers":
        return [float(cfg["eff"])] * len(lay)
    nl = 48
    return [I.layer_rank_schedule(li, nl) if li < nl else 0.10 for li in lay]


def make_train_inputs(torch, cfg, shapes, lay, device, seed, pool, sides=None):
    """`pool` independent sets of (X_i, G_i) per matrix and one W_i per
    matrix, drawn on the device: X_i = Z diag(sqrt(lambda)) Q_i^T (N x n,
    geometric spectrum at the matrix's effective rank, Q_i a shared Haar
    basis per width with permuted, sign-flipped rows), G_i = D X_i / N, W_i ~
    N(0, 0.02^2), in the configured dtypes.  For an output-side (Dobb-G)
    matrix X_i are output gradients (N x m) of the same recipe and G_i =
    X_i^T D / N."""
    import numpy as np
    from block_eigenbasis_preconditioning_gb300 import inputs as I
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    pdt = torch.bfloat16 if cfg["pdt"] == "bf16" else torch.float32
    adt = torch.bfloat16 if cfg["adt"] == "bf16" else torch.float32
    N = cfg["N"]
    effs = _eff_for(cfg, lay)
    lam_cache, haar_cache = {}, {}
    mix = []
    for i, (m, n) in enumerate(shapes):
        if sides is not None and sides[i] == "output":
            m, n = n, m
        key = (n, round(effs[i], 6))
        if key not in lam_cache:
            lam = I.geometric_spectrum(n, effs[i])
            lam = lam * (n / lam.sum())
            lam_cache[key] = torch.tensor(lam, dtype=torch.float32, device=device).sqrt_()
        if n not in haar_cache:
            haar_cache[n] = torch.tensor(I.haar_orthogonal(n, np.random.default_rng(seed + n)),
                                         dtype=torch.float32, device=device)
        perm = torch.randperm(n, generator=g, device=device)
        flip = torch.randint(0, 2, (n, 1), generator=g, device=device).float() * 2 - 1
        mix.append((lam_cache[key], perm, flip))
    Xsets = [[] for _ in range(pool)]
    Gsets = [[] for _ in range(pool)]
    Ws = []
    for i, (m, n) in enumerate(shapes):
        out = sides is not None and sides[i] == "output"
        mm, nn = (n, m) if out else (m, n)
        sq, perm, flip = mix[i]
        q = haar_cache[nn][perm] * flip
        for s in range(pool):
            Z = torch.randn(N, nn, generator=g, device=device)
            X = (Z * sq.unsqueeze(0)) @ q.T
            del Z
            D = torch.randn(mm, N, generator=g, device=device)
            G = (D @ X) / N
            del D
            Xsets[s].append(X.to(adt))
            Gsets[s].append((G.T if out else G).contiguous().to(pdt))
            del X, G
        W = torch.randn(mm, nn, generator=g, device=device) * 0.02
        Ws.append((W.T if out else W).contiguous().to(pdt))
        del q
    return Xsets, Gsets, Ws


def make_stress_moments(torch, shapes, B, device, seed, pool):
    """`pool` flat sets of block moments in the state's layout (matrix after
    matrix, B blocks of k x k each): A_b = Q diag(lambda) Q^T with Haar Q
    (QR of a Gaussian on the device, signs folded) and lambda log-spaced on
    [1e-6, 1] with +-1/4-spacing jitter, every relative gap >= 1e-3."""
    import numpy as np
    rng = np.random.default_rng(seed)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    total = sum(B * (n // B) ** 2 for _, n in shapes)
    sets = []
    for _ in range(pool):
        flat = torch.empty(total, dtype=torch.float32, device=device)
        off = 0
        for (m, n) in shapes:
            k = n // B
            for b in range(B):
                while True:
                    logs = np.linspace(0.0, -np.log(1e6), k)
                    if k > 2:
                        h = np.log(1e6) / (k - 1)
                        logs[1:-1] += rng.uniform(-0.25 * h, 0.25 * h, size=k - 2)
                    lam = np.exp(logs)
                    if k == 1 or (np.abs(np.diff(lam)) / lam[:-1]).min() >= 1e-3:
                        break
                Z = torch.randn(k, k, generator=g, device=device, dtype=torch.float64)
                q, r = torch.linalg.qr(Z)
                q = q * torch.sign(torch.diagonal(r)).unsqueeze(0)
                lt = torch.tensor(lam, dtype=torch.float64, device=device)
                a = (q * lt.unsqueeze(0)) @ q.T
                a = 0.5 * (a + a.T)
                flat[off:off + k * k] = a.reshape(-1).to(torch.float32)
                off += k * k
                del Z, q, r, a
        sets.append(flat)
    return sets


def _kernel_source_sha(name):
    p = os.path.join(ROOT, "block_eigenbasis_preconditioning_gb300", "csrc", name)
    try:
        with open(p, "rb") as f:
            return hashlib.sha256(f.read()).hexdigest()[:16]
    except OSError:
        return None


def _traffic_for(kernel_key, workload):
    """DRAM bytes per unit of work of that kernel (a launch, or for the
    eigensolver one refresh) from a committed ncu summary, if it was taken on
    the current sources of the kernel and on this workload."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)
        e = t.get(kernel_key)
        if e and e.get("workload") == workload and all(
                sha == _kernel_source_sha(src) for src, sha in e.get("sources", {}).items()):
            return e.get("bytes_per_unit")
    except Exception:
        pass
    return None


# ---------------------------------------------------------------------------
# CPU baseline: the oracle on a bounded sample
# ---------------------------------------------------------------------------

class OracleSample:
    """The fp64 oracle as it stands, on `layers_sample` layers of a workload
    (the same recipe, drawn on the host once): `step()` runs and times one
    accumulate (or, for the stress workloads, nothing), one refresh and one
    update, amortised like the GPU step (accumulate + update + refresh / T)."""

    def __init__(self, cfg_name="gpt2-xl", layers_sample=1, seed=0, basis="f32", refresh="eigh",
                 orth_steps=1, norm="sign", side="input"):
        import numpy as np
        from block_eigenbasis_preconditioning_gb300 import inputs as I
        from oracle import dobb as O
        self.cfg_name, self.refresh_method = cfg_name, refresh
        cfg = self.cfg = CONFIGS[cfg_name]
        rng = np.random.default_rng(seed)
        self.shapes, lay = model_shapes(cfg["model"], layers=layers_sample)
        self.params = sum(m * n for m, n in self.shapes)
        self.layers = layers_sample
        B = cfg["B"]
        self.orc = O.DobbOracle(self.shapes, B, BETA1, BETA2, refresh_period=0, scale_s=SCALE,
                                param_dtype=cfg["pdt"], eig_method="lapack", basis_dtype=basis,
                                refresh_method=refresh, orth_steps=orth_steps, norm=norm, side=side)
        self.Xs = None
        if cfg["kind"] == "train":
            effs = _eff_for(cfg, lay)
            bases = {}
            streams = []
            for (m, n), e in zip(self.shapes, effs):
                w = m if side == "output" else n
                if w not in bases:
                    bases[w] = I.haar_orthogonal(w, rng)
                streams.append(I.ActivationStream(w, e, rng, shared_basis=bases[w]))
            self.Xs = [s.draw(cfg["N"], rng, dtype=cfg["adt"]) for s in streams]
            if side == "output":
                self.Gs = [I.round_bf16_np(rng.standard_normal((m, n)).astype(np.float32) * 1e-3)
                           for m, n in self.shapes]
            else:
                self.Gs = [I.gradients_fp32(m, X, rng, dtype=cfg["pdt"])
                           for (m, _), X in zip(self.shapes, self.Xs)]
        else:
            for i, (m, n) in enumerate(self.shapes):
                k = n // B
                self.orc.A[i] = np.stack([I.spd_with_gap(k, rng, cond=1e6)[0] for _ in range(B)])
            self.Gs = [I.round_bf16_np(rng.standard_normal((m, n)).astype(np.float32) * 1e-3)
                       for m, n in self.shapes]
        self.Ws = [I.weights(m, n, rng, dtype=cfg["pdt"]) for m, n in self.shapes]
        self.seconds = None

    def step(self):
        t0 = time.perf_counter()
        if self.Xs is not None:
            self.orc.accumulate(self.Xs)
        t1 = time.perf_counter()
        self.orc.refresh()
        t2 = time.perf_counter()
        self.Ws = self.orc.step(self.Ws, self.Gs, LR)
        t3 = time.perf_counter()
        acc, ref, upd = t1 - t0, t2 - t1, t3 - t2
        self.seconds = {"accumulate": acc, "refresh": ref, "update": upd}
        return self.params / (acc + upd + ref / self.cfg["T"])

    def describe(self):
        return (f"{self.layers} {self.cfg['model']} layer(s) of the {self.cfg_name} workload "
                f"({self.params} params, {len(self.shapes)} matrices, the same input recipe drawn "
                f"once on the host): per step one accumulate + one "
                f"{'LAPACK' if self.refresh_method == 'eigh' else 'orthogonal-iteration'} refresh "
                f"+ one update in fp64 numpy, amortised as accumulate + update + "
                f"refresh/{self.cfg['T']}")


def cpu_baseline(cfg_name="gpt2-xl", layers_sample=1, **kw):
    s = OracleSample(cfg_name, layers_sample, **kw)
    v = s.step()
    return {"value": v, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": s.describe(), "seconds": s.seconds}


def workload_name(cfg_name, cfg, n_matrices, params, layers):
    base = {"gpt2-xl": "gpt2-xl", "gpt2-small": "gpt2-small", "single": "single 768x768",
            "llama3-8b": "llama3-8b"}[cfg["model"]]
    if cfg["kind"] == "stress":
        return (f"refresh stress on gpt2-xl shapes B={cfg['B']}: {n_matrices} matrices, {params} "
                f"params; a step sets every block's moments to a fresh SPD block (gap >= 1e-3, "
                f"cond 1e6) and eigensolves every block (no parameter update)")
    s = (f"{base} B={cfg['B']}: {n_matrices} matrices, {params:.4g} params, {cfg['pdt']} W/G, "
         f"fp32 M, X {cfg['N']} {cfg['adt']} tokens/matrix, refresh every {cfg['T']}")
    if layers is not None:
        s += f" (first {layers} layers)"
    return s


def run_reference(args):
    rank, world, _ = _env_rank()
    if rank != 0:
        return 0
    cfg = CONFIGS[args.config]
    shapes, _ = model_shapes(cfg["model"], args.layers)
    params = sum(m * n for m, n in shapes)
    sample = OracleSample(args.config, 1, basis=args.basis, refresh=args.refresh,
                          orth_steps=args.orth_steps, norm=args.norm, side=args.side)
    for _ in range(args.warmup):
        sample.step()
    steps = [sample.step() for _ in range(max(1, args.steps))]
    v = sorted(steps)[len(steps) // 2]
    name = workload_name(args.config, cfg, len(shapes), params, args.layers)
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": params / v * 1e3 if v else None,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": f"{name}; timed on the oracle sample: {sample.describe()}",
                       "B": cfg["B"], "refresh_period": cfg["T"], "tokens": cfg["N"],
                       "parallelism": "host cores"},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                             "sample": sample.describe()},
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
    from block_eigenbasis_preconditioning_gb300.sharding import partition_matrices

    rank, world, local = _env_rank()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    cfg = dict(CONFIGS[args.config])
    if args.pool is not None:
        cfg["pool"] = args.pool
    all_shapes, all_lay = model_shapes(cfg["model"], args.layers)
    total_params = sum(m * n for m, n in all_shapes)
    # N > 1: whole matrices placed on ranks, no collective on the data path
    mine = partition_matrices(all_shapes, cfg["B"], world, max(cfg["N"], 1), cfg["T"])[rank]
    shapes = [all_shapes[i] for i in mine]
    lay = [all_lay[i] for i in mine]
    B, T = cfg["B"], cfg["T"]
    # Dobb-G blocks the output axis of every layer matrix; a matrix whose m
    # does not split into B blocks stays on the input side
    sides = [("output" if args.side == "output" and m % B == 0 and m // B <= 1024 else "input")
             for m, n in shapes]
    peaks = probe_peaks(torch) if not args.no_probe else None
    torch.manual_seed(1234 + rank)
    stress = cfg["kind"] == "stress"
    if stress:
        Msets = make_stress_moments(torch, shapes, B, device, seed=1234 + rank, pool=cfg["pool"])
        g = torch.Generator(device=device)
        g.manual_seed(99 + rank)
        Gsets = [[(torch.randn(m, n, generator=g, device=device) * 1e-3).to(torch.bfloat16)
                  for m, n in shapes]]
        Ws = [(torch.randn(m, n, generator=g, device=device) * 0.02).to(torch.bfloat16)
              for m, n in shapes]
        Xsets = None
    else:
        Xsets, Gsets, Ws = make_train_inputs(torch, cfg, shapes, lay, device, seed=1234 + rank,
                                             pool=cfg["pool"], sides=sides)
    opt = Dobb(shapes, B, BETA1, BETA2, refresh_period=T, scale_s=SCALE,
               param_dtype=cfg["pdt"], act_dtype=cfg["adt"], device=device,
               basis_dtype=args.basis, refresh=args.refresh, orth_steps=args.orth_steps,
               norm=args.norm, side=sides)
    stream = torch.cuda.current_stream()
    moments = opt.tensor("moments")

    stress_t = [0]   # the stress workload's own step counter (it runs no optimizer step)

    def one_step(t, ev=None):
        if stress:
            t = stress_t[0]
            stress_t[0] += 1
        s = t % cfg["pool"]
        if ev is not None:
            ev[0].record(stream)
        if stress:
            moments.copy_(Msets[s])
        else:
            opt.accumulate(Xsets[s])
        if ev is not None:
            ev[1].record(stream)
        if stress:
            opt.refresh()   # the stress workload: every block of every matrix, every step
        else:
            opt.step(Ws, Gsets[s % len(Gsets)], LR)
        if ev is not None:
            ev[2].record(stream)

    # warm-up: the first step refreshes from the identity (cold); time it
    cold_ms = None
    for w in range(args.warmup):
        if w == 0 and opt.t % T == 0:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            if stress:
                moments.copy_(Msets[0])
                stress_t[0] += 1
            else:
                opt.accumulate(Xsets[0])
            e0.record(stream)
            opt.refresh()
            e1.record(stream)
            torch.cuda.synchronize()
            cold_ms = e0.elapsed_time(e1)
            if not stress:
                opt.step(Ws, Gsets[0], LR)   # its scheduled refresh runs warm from the cold result
            continue
        one_step(opt.t)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()

    # timed region
    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    is_refresh = []
    props = torch.cuda.get_device_properties(device)
    clocks = ClockSampler(str(getattr(props, "uuid", "")) or None)
    clocks.start()
    launches0 = opt.launch_count
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    start.record(stream)
    for i in range(K):
        t = opt.t
        is_refresh.append(T > 0 and t % T == 0)
        one_step(t, evs[i])
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
    mean = lambda v: sum(v) / len(v) if v else None
    acc_ms = [evs[i][0].elapsed_time(evs[i][1]) for i in range(K)]
    upd_ref_ms = [evs[i][1].elapsed_time(evs[i][2]) for i in range(K)]
    upd_ms = [v for v, r in zip(upd_ref_ms, is_refresh) if not r]
    ref_steps = [v for v, r in zip(upd_ref_ms, is_refresh) if r]
    upd_mean = mean(upd_ms)
    refresh_ms = None
    if stress:
        refresh_ms = mean(upd_ref_ms)    # a stress step is the refresh alone
    elif ref_steps and upd_mean is not None:
        refresh_ms = mean(ref_steps) - upd_mean
    # the update alone when every timed step refreshes (stress), and the
    # refresh alone when the timed window held none
    if not stress and (upd_mean is None or refresh_ms is None):
        e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        saved_t = opt.t
        opt.t = 1 if T != 1 else 0
        e0.record(stream)
        opt.refresh()
        e1.record(stream)
        if T == 1:
            opt.set_refresh_period(0)
        opt.step(Ws, Gsets[0], LR)
        e2.record(stream)
        torch.cuda.synchronize()
        opt.t = saved_t
        if refresh_ms is None:
            refresh_ms = e0.elapsed_time(e1)
        if upd_mean is None:
            upd_mean = e1.elapsed_time(e2)
        if T == 1:
            opt.set_refresh_period(1)

    mp = _measured_peaks()
    hbm = mp["hbm_gbs"]
    wm = work_model(shapes, B, max(cfg["N"], 0), pbytes=2 if cfg["pdt"] == "bf16" else 4,
                    xbytes=2 if cfg["adt"] == "bf16" else 4, refresh=args.refresh,
                    orth_steps=args.orth_steps, norm=args.norm, sides=sides)
    if stress:
        wm["acc_bytes"] = 8 * sum(B * (n // B) ** 2 for _, n in shapes)   # moment copy r + w
        wm["acc_flops"] = 0
    ffma_peak = peaks["ffma_tflops"] if peaks else 152 * 128 * 2 * 2.07e9 / 1e12
    ffma_src = peaks["source"] + " (FFMA)" if peaks else "nominal unit count (probes skipped)"
    ffma_update = args.norm != "sign"
    phases = {
        "update": None if stress else
                  {"ms": upd_mean, "kernel": "step_ffma_kernel" if ffma_update else "step_tc_kernel",
                   "bound": "hbm", "achieved": wm["update_bytes"] / (upd_mean * 1e-3) / 1e9,
                   "peak": hbm, "peak_source": mp["source"], "unit": "GB/s",
                   "flops": wm["update_flops"], "bytes": wm["update_bytes"]},
        "accumulate": {"ms": mean(acc_ms), "kernel": "syrk_tc_kernel" if not stress else "moment copy",
                       "bound": "hbm", "achieved": wm["acc_bytes"] / (mean(acc_ms) * 1e-3) / 1e9,
                       "peak": hbm, "peak_source": mp["source"], "unit": "GB/s",
                       "flops": wm["acc_flops"], "bytes": wm["acc_bytes"]},
        "refresh": {"ms": refresh_ms, "cold_ms": cold_ms,
                    "kernel": ("grid eigensolver (gj_* kernels)" if args.refresh == "eigh"
                               else "orth_kernel"),
                    "unit_of_work": "one refresh of every block (all its launches)",
                    "bound": "alu", "achieved": wm["refresh_flops"] / (refresh_ms * 1e-3) / 1e12,
                    "peak": ffma_peak, "peak_source": ffma_src, "unit": "TFLOP/s",
                    "flops": wm["refresh_flops"]},
    }
    phases = {k: v for k, v in phases.items() if v is not None}
    for p in phases.values():
        p["frac"] = p["achieved"] / p["peak"] if p.get("achieved") else None
    # dominant kernel: most device time per refresh cycle
    per_cycle = max(T, 1)
    share = {"accumulate": mean(acc_ms) * per_cycle, "refresh": refresh_ms}
    if not stress:
        share["update"] = upd_mean * per_cycle
    dom = max(share, key=share.get)
    d = phases[dom]
    wl = workload_name(args.config, cfg, len(all_shapes), total_params, args.layers)
    roofline = {"bound": d["bound"], "achieved": d["achieved"], "peak": d["peak"], "unit": d["unit"],
                "frac": d["frac"], "traffic": _traffic_for(d["kernel"], args.config),
                "kernel": d["kernel"], "peak_source": d["peak_source"]}
    # whole-step roofline: HBM bytes at the copy rate plus the refresh flops at
    # the FFMA rate, amortised over the refresh period
    floor_ms = ((0 if stress else wm["update_bytes"]) + wm["acc_bytes"]) / (hbm * 1e9) * 1e3 + \
        wm["refresh_flops"] / (ffma_peak * 1e12) * 1e3 / per_cycle

    e2e = None
    if not args.no_e2e and not stress:
        e2e = run_e2e(torch, opt, cfg, shapes, lay, sides, Ws, K, stream, total_params, world)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        try:
            cpu = cpu_baseline(args.config, basis=args.basis, refresh=args.refresh,
                               orth_steps=args.orth_steps, norm=args.norm, side=args.side)
        except Exception as ex:  # pragma: no cover
            cpu = {"error": repr(ex)}

    if rank == 0:
        amort = mean(acc_ms) + (0 if stress else upd_mean) + refresh_ms / per_cycle
        line = {"metric": METRIC, "value": total_params / (ms_step * 1e-3), "unit": UNIT,
                "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": ms_step,
                "higher_is_better": True, "scaling": "strong" if world > 1 else "weak",
                "vs_baseline": None, "dtype": "f32", "data": "synthetic",
                "config": {"workload": wl, "B": B, "refresh_period": T, "tokens": cfg["N"],
                           "basis": args.basis, "norm": args.norm, "side": args.side,
                           "refresh": args.refresh if args.refresh == "eigh" else f"orth x{args.orth_steps}",
                           "input_pool": f"{cfg['pool']} independently drawn input sets, step t "
                                         f"uses set t mod {cfg['pool']}",
                           "l2": "inputs larger than L2 (every step streams its own set)",
                           "refresh_steps_timed": sum(is_refresh),
                           "parallelism": (f"{world} GPUs, whole matrices placed per rank, no "
                                           f"collective" if world > 1 else "single GPU")},
                "phases_ms": {"accumulate": mean(acc_ms), "update": upd_mean, "refresh": refresh_ms,
                              "refresh_cold": cold_ms, "amortized_step": amort},
                "phases": phases, "roofline": roofline,
                "step_roofline": {"floor_ms": floor_ms, "frac": floor_ms / ms_step,
                                  "note": "(update + moment bytes) / HBM copy rate + refresh "
                                          "9k^3 flops / FFMA rate / T"},
                "peaks": dict(peaks or {}, hbm_gbs=hbm, bf16_tflops=mp["bf16_tflops"],
                              measured_source=mp["source"]),
                "clocks": clk, "gpu_launches": launches, "e2e": e2e, "cpu_baseline": cpu}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def _flat(torch, like, device=None, pin=False):
    """One flat buffer with room for tensors shaped like `like` (one dtype),
    each view starting on a 256-byte boundary; returns (buffer, views)."""
    esz = like[0].element_size()
    align = max(1, 256 // esz)
    offs, tot = [], 0
    for t in like:
        offs.append(tot)
        tot += (t.numel() + align - 1) // align * align
    if pin:
        buf = torch.empty(tot, dtype=like[0].dtype).pin_memory()
    else:
        buf = torch.empty(tot, dtype=like[0].dtype, device=device)
    views = [buf[o:o + t.numel()].view(t.shape) for o, t in zip(offs, like)]
    return buf, views


def _bind_to_gpu_local_cpus(torch):
    """Run this process on the host cores attached to the current GPU, so that
    pinned buffers allocated meanwhile land in that socket's memory (a
    buffer on the other socket crosses the socket link on every copy).
    Returns the previous affinity; best effort on systems that do not expose
    the GPU's local CPUs."""
    prev = os.sched_getaffinity(0)
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
    return prev


def run_e2e(torch, opt, cfg, shapes, lay, sides, W, K, stream, params, world):
    """End to end through the public API with host buffers.  Every step
    copies that step's activations and gradients from pinned host memory
    (two independently drawn host sets, alternating) and copies the updated
    parameters back to pinned host memory; the inputs and parameters of all
    matrices sit in one flat buffer per kind (a flat parameter buffer, as a
    training loop keeps them).  The input copies of step i+1 run during step i
    (double-buffered device inputs): the activations in two halves on two copy
    streams, then the gradients; the parameter copy of step i runs on a third
    stream during step i+1's accumulate, and step i+1's update waits for it."""
    dev = W[0].device
    Xs2, Gs2, _ = make_train_inputs(torch, dict(cfg, pool=2), shapes, lay, dev, seed=777,
                                    pool=2, sides=sides)
    prev_cpus = _bind_to_gpu_local_cpus(torch)
    Xh, Gh = [], []
    for s2 in range(2):
        hb, hv = _flat(torch, Xs2[s2], pin=True)
        for v, x in zip(hv, Xs2[s2]):
            v.copy_(x)
        Xh.append(hb)
        hb, hv = _flat(torch, Gs2[s2], pin=True)
        for v, g in zip(hv, Gs2[s2]):
            g_ = g
            v.copy_(g_)
        Gh.append(hb)
    Xd = [_flat(torch, Xs2[0], device=dev) for _ in range(2)]
    Gd = [_flat(torch, Gs2[0], device=dev) for _ in range(2)]
    del Xs2, Gs2
    Wd_buf, Wd = _flat(torch, W, device=dev)
    for v, w in zip(Wd, W):
        v.copy_(w)
    Wh = torch.empty_like(Wd_buf, device="cpu").pin_memory()
    link = host_link_rates(torch)
    os.sched_setaffinity(0, prev_cpus)
    # the rate of one copy of a step's flat activation buffer (best of 3)
    best = 0.0
    for _ in range(3):
        ef0, ef1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        ef0.record(stream)
        Xd[0][0].copy_(Xh[0], non_blocking=True)
        ef1.record(stream)
        torch.cuda.synchronize()
        best = max(best, Xh[0].numel() * Xh[0].element_size() / (ef0.elapsed_time(ef1) * 1e-3) / 1e9)
    link["h2d_flat_x_gbs"] = best
    h2d = Xh[0].numel() * Xh[0].element_size() + Gh[0].numel() * Gh[0].element_size()
    d2h = Wh.numel() * Wh.element_size()
    cx, cg, cw = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    x_done = [torch.cuda.Event() for _ in range(2)]
    g_done = [torch.cuda.Event() for _ in range(2)]
    x_used = [torch.cuda.Event() for _ in range(2)]
    g_used = [torch.cuda.Event() for _ in range(2)]
    w_ready, w_out = torch.cuda.Event(), torch.cuda.Event()

    half_done = [torch.cuda.Event() for _ in range(2)]

    def issue(i):
        # the activations in two halves on two copy streams (one large copy
        # alone runs well below the link rate), then the gradients
        b = i % 2
        if i >= 2:
            cx.wait_event(x_used[b])
            cx.wait_event(g_used[b])
            cg.wait_event(x_used[b])
        h = Xh[b].numel() // 2
        with torch.cuda.stream(cg):
            Xd[b][0][h:].copy_(Xh[b][h:], non_blocking=True)
        half_done[b].record(cg)
        with torch.cuda.stream(cx):
            Xd[b][0][:h].copy_(Xh[b][:h], non_blocking=True)
        cx.wait_event(half_done[b])
        x_done[b].record(cx)
        with torch.cuda.stream(cx):
            Gd[b][0].copy_(Gh[b], non_blocking=True)
        g_done[b].record(cx)

    torch.cuda.synchronize()
    t0 = time.perf_counter()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for cs in (cx, cg, cw):
        cs.wait_stream(stream)
    issue(0)
    if K > 1:
        issue(1)
    for i in range(K):
        b = i % 2
        stream.wait_event(x_done[b])
        opt.accumulate(Xd[b][1])
        x_used[b].record(stream)
        stream.wait_event(g_done[b])
        if i > 0:
            stream.wait_event(w_out)      # the previous step's parameters have left
        opt.step(Wd, Gd[b][1], LR)
        g_used[b].record(stream)
        w_ready.record(stream)
        cw.wait_event(w_ready)
        with torch.cuda.stream(cw):
            Wh.copy_(Wd_buf, non_blocking=True)
        w_out.record(cw)
        if i + 2 < K:
            issue(i + 2)
    stream.wait_event(w_out)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / K
    return {"value": params / (ms * 1e-3), "unit": UNIT, "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "wall_ms_per_step": (time.perf_counter() - t0) * 1e3 / K,
            "host_link": link,
            "copy_floor_ms": max(h2d / (link["h2d_gbs"] * 1e9), d2h / (link["d2h_gbs"] * 1e9)) * 1e3,
            "overlap": "inputs of step i+1 copied during step i (activations in two halves on two "
                       "streams, then gradients); parameters of step i copied back during step i+1's "
                       "accumulate; one flat buffer per kind"}


def _relaunch_distributed(args):
    """`--gpus N` without a launcher: run this script under torch's launcher
    with N processes on this node."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={args.gpus}", "--master-addr", "127.0.0.1",
           "--master-port", str(29500 + os.getpid() % 1000), os.path.abspath(__file__)] + \
        [a for a in sys.argv[1:]]
    return subprocess.call(cmd)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--config", default="gpt2-xl", choices=sorted(CONFIGS))
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--pool", type=int, default=None, help="input sets in the device pool")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-probe", action="store_true")
    ap.add_argument("--refresh", default="eigh", choices=["eigh", "orth"],
                    help="eigh: complete eigendecomposition; orth: orthogonal iteration with "
                         "Cholesky QR (the pages' principal refresh)")
    ap.add_argument("--orth-steps", type=int, default=1)
    ap.add_argument("--norm", default="sign", choices=["sign", "l2"],
                    help="coefficient normalisation: sign (Dobb) or l2 (Dobb-l2)")
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
    rank, world, _ = _env_rank()
    if args.gpus > 1 and world == 1 and "RANK" not in os.environ:
        return _relaunch_distributed(args)
    if world > 1 and args.gpus != world:
        print(json.dumps({"error": f"--gpus {args.gpus} but WORLD_SIZE {world}"}), flush=True)
        return 2
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
