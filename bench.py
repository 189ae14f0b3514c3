"""Throughput of the per-shard mixed-precision ZeRO optimizer step on GB300.

Default workload: the per-tensor (non-flat, multi-tensor-apply) list of the
Llama-3-8B shapes -- the 128256x4096 embedding plus 8 decoder layers (q 4096x4096,
k/v 1024x4096, o 4096x4096, gate/up 14336x4096, down 4096x14336, two 4096
RMSNorm weights): 73 tensors, 2,270,232,576 parameters, bf16 gradients
~N(0, 1e-3), fp32 masters ~N(0, 0.02), AdamW lr 1e-4 wd 0.1, global L2 clip
1.0.  It is the largest workload that fits one GPU (36 GB of state and
gradients, 63.6 GB of algorithmic traffic per step).  Inputs are synthetic and
seeded and are resident in HBM before the timed region; they are far larger
than L2, so no L2 flush is needed.

One "step" is one call of zero_opt_step (zero_opt_step_tensors for the list):
pass 1 (reduce, overflow flag, sum of squares, decision) and pass 2 (unscale,
clip, AdamW, 16-bit copy).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload pertensor|gpt2|gpt2_master16|llama|fused]

Prints one JSON line (rank 0).  Under torchrun with N > 1 ranks it times the
sharded ZeRO-2 step of the same model over the N GPUs (strong scaling: each
rank owns 1/N of the parameters; all-to-all of the gradient bytes, statistics
folded on the device, all-gather of the 16-bit parameters; --zero3 keeps them
sharded), the timing being the maximum over ranks; --replicas instead runs an
independent copy of the one-GPU workload per rank (weak scaling).  --zero2 /
--zero3 select the sharded step on one GPU too.  --impl reference times the
CPU oracle (single-threaded C++) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "optimizer-step params/s and achieved HBM GB/s (% of GB300 peak), 1 GPU"
FALLBACK_HBM_GBS = 6800.0


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------- workloads

def llama_shapes(div=1):
    """Embedding plus 8 decoder layers of Llama-3-8B; every dimension divided
    by `div` for scaled-down profiling captures (1: the workload itself)."""
    H, KV, F, V = 4096 // div, 1024 // div, 14336 // div, 128256 // div
    shapes = [(V, H)]
    for _ in range(8):
        shapes += [(H, H), (KV, H), (KV, H), (H, H), (F, H), (F, H), (H, F), (H,), (H,)]
    return shapes


WORKLOADS = {
    "gpt2": dict(desc="GPT-2-small-sized flat buffer, 124,439,808 params, N=1, bf16 grads "
                      "~N(0,1e-2), AdamW lr 3e-4 wd 0.01, global L2 clip 1.0, no loss scaling",
                 numel=124_439_808, world=1, R=1, K=1, dtype="bf16", lr=3e-4, wd=0.01,
                 clip=1.0, dynamic=False, scale=1.0, sigma=1e-2, seed=0x5EED0002),
    "llama": dict(desc="Llama-3-8B ZeRO-2 shard: rank 0 of N=8 over 8,030,261,248 params "
                       "(1,003,782,656-param shard), fp16 grads ~N(0,1e-4) x dynamic scale 2^16, "
                       "window 1000, AdamW lr 1e-4 wd 0.1",
                  numel=8_030_261_248, world=8, R=1, K=1, dtype="fp16", lr=1e-4, wd=0.1,
                  clip=0.0, dynamic=True, scale=65536.0, sigma=1e-4, seed=0x5EED0003),
    "fused": dict(desc="fused local rank reduction + step: 250,000,000-param shard, 8 ranks x "
                       "4 micro-steps of fp16 grads ~N(0,1e-3) x 1024, divided by 32, AdamW lr "
                       "2e-4 wd 0.01, clip 1.0",
                  numel=250_000_000, world=1, R=8, K=4, dtype="fp16", lr=2e-4, wd=0.01,
                  clip=1.0, dynamic=False, scale=1024.0, sigma=1e-3, seed=0x5EED0004),
    "gpt2_master16": dict(desc="GPT-2-small-sized flat buffer, 124,439,808 params, N=1, bf16 grads "
                               "~N(0,1e-2), bf16 low-precision master weights (no fp32 master), "
                               "AdamW lr 3e-4 wd 0.01, global L2 clip 1.0, no loss scaling",
                          numel=124_439_808, world=1, R=1, K=1, dtype="bf16", lr=3e-4, wd=0.01,
                          clip=1.0, dynamic=False, scale=1.0, sigma=1e-2, seed=0x5EED0002,
                          master16=True),
    "pertensor": dict(desc="per-tensor list: Llama-3-8B embedding + 8 decoder layers, 73 "
                           "tensors, 2,270,232,576 params, bf16 grads ~N(0,1e-3), AdamW lr 1e-4 "
                           "wd 0.1, clip 1.0",
                      numel=2_270_232_576, world=1, R=1, K=1, dtype="bf16", lr=1e-4, wd=0.1,
                      clip=1.0, dynamic=False, scale=1.0, sigma=1e-3, seed=0x5EED0005),
}


# Committed ncu summaries of one pass-2 launch per workload, from which the
# per-parameter DRAM traffic is read (times the workload's parameter count;
# the per-tensor list's was captured at its full size, GPT-2's at 100M
# parameters: the kernel streams, so its traffic is proportional to the
# elements).
PASS2_PROFILES = {
    "gpt2": "pass2_kernel_gpt2_100M_ncu_full.md",
    "pertensor": "pass2_kernel_pertensor_full_dram.md",
}


def pass2_traffic_per_param(workload):
    """(DRAM bytes per parameter of one pass-2 launch, profile file) from the
    committed ncu summary of this workload, or (None, None) when there is none
    or the pass-2 kernel source changed since the capture."""
    import hashlib
    import re
    name = PASS2_PROFILES.get(workload)
    if name is None:
        return None, None
    try:
        prof = open(os.path.join(ROOT, "profiles", name)).read()
        src = open(os.path.join(ROOT, "zero_sharded_mixed_05_gb300", "csrc", "kernels.cuh")).read()
    except OSError:
        return None, None
    a = src.find("// ------------------------------------------------------------- pass 2")
    b = src.find("// ------------------------------------------------------------- 16-bit copy")
    mt = re.search(r"traffic_bytes_per_param: ([0-9.]+)", prof)
    mh = re.search(r"pass2_source_sha256: ([0-9a-f]{64})", prof)
    if a < 0 or b < 0 or not mt or not mh:
        return None, None
    if hashlib.sha256(src[a:b].encode()).hexdigest() != mh.group(1):
        return None, None
    return float(mt.group(1)), "profiles/" + name


def state_bytes_per_param(w):
    # fp32 master/m/v read + written + 16-bit copy written (26 B); with 16-bit
    # masters: 16-bit master read, m/v read + written, 16-bit master written (20 B)
    return 20 if w.get("master16") else 26


def algorithmic_bytes_per_param(w):
    # R*K 16-bit gradient reads + the optimizer state traffic
    return 2 * w["R"] * w["K"] + state_bytes_per_param(w)


def pass2_bytes_per_param(w, stash):
    # pass 2 alone: gradients (or the fp32 stash) read, state read and written, copy written
    return (4 if stash else 2 * w["R"] * w["K"]) + state_bytes_per_param(w)


class Setup:
    """Device buffers of one workload, filled by the seeded generator."""

    def __init__(self, name, device):
        import torch

        import synth
        import zero_sharded_mixed_05_gb300 as z
        w = WORKLOADS[name]
        self.w, self.name, self.z = w, name, z
        code = z.FP16 if w["dtype"] == "fp16" else z.BF16
        tdt = torch.float16 if code == z.FP16 else torch.bfloat16
        kind = synth.F16 if code == z.FP16 else synth.BF16
        self.tdt = tdt
        cfg = z.make_config(numel=w["numel"], world=w["world"], grad_dtype=code, lr=w["lr"],
                            weight_decay=w["wd"], max_grad_norm=w["clip"],
                            dynamic_scale=w["dynamic"], init_scale=w["scale"],
                            scale_window=1000, master16=w.get("master16", False))
        self.h = z.zero_opt_create(cfg)
        nb = w["R"] * w["K"]
        self.stash = None
        if name == "pertensor":
            shapes = llama_shapes(w.get("div", 1))
            self.items, off = [], 0
            for shp in shapes:
                n = int(np.prod(shp))
                master = torch.empty(n, dtype=torch.float32, device=device)
                synth.fill_gpu(master, w["seed"], 0, off, 0.02, synth.F32)
                g = torch.empty(n, dtype=tdt, device=device)
                synth.fill_gpu(g, w["seed"], 1, off, w["sigma"] * w["scale"], kind)
                self.items.append(dict(numel=n, master=master,
                                       m=torch.zeros(n, device=device),
                                       v=torch.zeros(n, device=device),
                                       param16=master.to(tdt), grads=[g]))
                off += n
            self.n = off
            self.lst = z.make_tensor_list(self.items)
            self.grads = [it["grads"][0] for it in self.items]
            self.p16 = [it["param16"] for it in self.items]
        else:
            b, e, S, P = z.zero_opt_shard_bounds(self.h, 0)
            self.n = e - b
            n = self.n
            self.master = torch.empty(n, dtype=torch.float32, device=device)
            synth.fill_gpu(self.master, w["seed"], 0, b, 0.02, synth.F32)
            self.m = torch.zeros(n, device=device)
            self.v = torch.zeros(n, device=device)
            # ZeRO-2 keeps the full 16-bit parameter buffer; the step writes its slice
            self.p16_full = torch.zeros(P, dtype=tdt, device=device)
            self.p16_full[b:e].copy_(self.master)
            self.grads = []
            for i in range(nb):
                g = torch.empty(n, dtype=tdt, device=device)   # shard-local (reduce-scattered)
                synth.fill_gpu(g, w["seed"], 1 + i, b, w["sigma"] * w["scale"], kind)
                self.grads.append(g)
            if nb > 4:
                self.stash = torch.empty(n, dtype=torch.float32, device=device)
            if w.get("master16"):
                self.master = None        # the 16-bit parameters are the masters
            self.bufs = z.make_buffers(self.master, self.m, self.v, self.p16_full, self.grads,
                                       n_ranks=w["R"], n_micro=w["K"], grads_shard_local=True,
                                       stash=self.stash)
            self.p16 = [self.p16_full[b:e]]
        torch.cuda.synchronize()

    def alternate_buffers(self):
        """Two (gradients, 16-bit parameter views, step function) sets that
        share the optimizer state: the workload's own buffers and a second
        copy of the gradient and 16-bit parameter buffers."""
        import torch
        z = self.z
        g2 = [torch.empty_like(g) for g in self.grads]
        if self.name == "pertensor":
            items2 = [dict(it, grads=[g], param16=torch.empty_like(it["param16"]))
                      for it, g in zip(self.items, g2)]
            lst2 = z.make_tensor_list(items2)
            p2 = [it["param16"] for it in items2]
            return [(self.grads, self.p16, self.step),
                    (g2, p2, lambda sp, lst2=lst2: z.zero_opt_step_tensors(self.h, 0, lst2, sp))]
        w = self.w
        # with 16-bit masters the parameters are optimizer state: one buffer
        p16b = self.p16_full if w.get("master16") else torch.empty_like(self.p16_full)
        bufs2 = z.make_buffers(self.master, self.m, self.v, p16b, g2, n_ranks=w["R"],
                               n_micro=w["K"], grads_shard_local=True, stash=self.stash)
        b, e, _, _ = z.zero_opt_shard_bounds(self.h, 0)
        return [(self.grads, self.p16, self.step),
                (g2, [p16b[b:e]], lambda sp, bufs2=bufs2: z.zero_opt_step(self.h, 0, bufs2, sp))]

    def step(self, stream=None):
        if self.name == "pertensor":
            self.z.zero_opt_step_tensors(self.h, 0, self.lst, stream)
        else:
            self.z.zero_opt_step(self.h, 0, self.bufs, stream)

    def input_bytes(self):
        return sum(g.numel() * g.element_size() for g in self.grads)

    def output_bytes(self):
        return sum(p.numel() * p.element_size() for p in self.p16)


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.idx)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((ts, parts))
        inside = [p for ts, p in rows if t0 - 0.15 <= ts <= t1 + 0.15] or [p for _, p in rows]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[1]) for p in inside if num(p[1]) is not None]
        mx = [num(p[2]) for p in inside if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i in range(4)
                          if p[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside),
                "power_w_max": max((num(p[3]) or 0.0) for p in inside)}


# ---------------------------------------------------------------- arms

def emit(line):
    """Print the bench's JSON line as the last line of stdout: anything a
    native library (NCCL's version banner) left in the C stdio buffer is
    flushed first."""
    import ctypes
    sys.stdout.flush()
    try:
        ctypes.CDLL(None).fflush(None)
    except (OSError, AttributeError):
        pass
    print(json.dumps(line), flush=True)


def max_over_ranks(value: float, device) -> float:
    """Largest value over the ranks of the default process group."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class OracleSample:
    """The single-threaded C++ oracle on a contiguous sample of the workload
    (same generator, same hyper-parameters); inputs are generated once."""

    def __init__(self, name, elems=4_000_000):
        import oracle as O
        import synth
        w = WORKLOADS[name]
        self.O = O
        self.code = O.FP16 if w["dtype"] == "fp16" else O.BF16
        kind = synth.F16 if self.code == O.FP16 else synth.BF16
        self.nb = w["R"] * w["K"]
        self.n = n = min(w["numel"] // w["world"], max(elems // self.nb, 1))
        self.master = synth.normal_np(w["seed"], 0, 0, n, 0.02, synth.F32)
        self.grads = [synth.normal_np(w["seed"], 1 + i, 0, n, w["sigma"] * w["scale"], kind)
                      for i in range(self.nb)]
        self.m = np.zeros(n, np.float32)
        self.v = np.zeros(n, np.float32)
        self.p16 = np.zeros(n, np.uint16)
        self.hp = O.hparams(lr=w["lr"], weight_decay=w["wd"], max_grad_norm=w["clip"],
                            dynamic_scale=w["dynamic"])
        self.st = O.scaler(w["scale"])
        self.total_steps = 0
        self.total_s = 0.0

    def rate(self, budget_s):
        """Params/s over oracle steps run for about budget_s seconds."""
        steps = 0
        t0 = time.perf_counter()
        while True:
            self.O.step(self.hp, self.st, self.grads, self.code, self.master, self.m, self.v,
                        self.p16, self.code, float(self.nb))
            steps += 1
            el = time.perf_counter() - t0
            if el >= budget_s:
                break
        self.total_steps += steps
        self.total_s += el
        return self.n * steps / el

    def info(self):
        return dict(kind="oracle", cores=1,
                    sample=f"{self.total_steps} oracle steps over the first {self.n:,} "
                           f"parameters of the workload ({self.nb} gradient buffer(s)), "
                           f"{self.total_s:.1f} s of CPU time")


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    name = args.workload
    sample = OracleSample(name)
    for _ in range(args.warmup):
        sample.rate(0.05)
    sample.total_steps, sample.total_s = 0, 0.0
    per_step = max(0.05, min(5.0, 60.0 / max(args.steps, 1)))
    rates = [sample.rate(per_step) for _ in range(args.steps)]
    value = statistics.median(rates)
    w = WORKLOADS[name]
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "params/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * (w["numel"] // w["world"]) / value,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded SplitMix64 / Irwin-Hall)",
            "config": {"workload": w["desc"], "params": w["numel"] // w["world"]},
            "cpu_baseline": {"value": value, "unit": "params/s", **sample.info()},
            "e2e": {"value": value, "unit": "params/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    emit(line)
    return 0


def e2e_pipelined(setup, compute, steps):
    """Milliseconds per step of H2D(grads) -> step -> D2H(16-bit params) with
    double-buffered device buffers and separate copy streams."""
    import torch
    host_g = [torch.empty(g.shape, dtype=g.dtype, pin_memory=True) for g in setup.grads]
    for hg, g in zip(host_g, setup.grads):
        hg.copy_(g)
    host_p = [torch.empty(p.shape, dtype=p.dtype, pin_memory=True) for p in setup.p16]
    sets = setup.alternate_buffers()           # [(grads, p16 views, step fn)] x 2
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()            # noqa: E731
    up = [ev(), ev()]
    done = [ev(), ev()]
    down = [None, None]
    sp = compute.cuda_stream

    def run(k):
        start = torch.cuda.Event(enable_timing=True)
        stop = torch.cuda.Event(enable_timing=True)
        start.record(compute)
        h2d.wait_event(start)
        with torch.cuda.stream(h2d):
            for hg, g in zip(host_g, sets[0][0]):
                g.copy_(hg, non_blocking=True)
        up[0].record(h2d)
        for i in range(k):
            b = i % 2
            if i + 1 < k:                      # upload the next step's gradients
                if i >= 1:
                    h2d.wait_event(done[1 - b])
                with torch.cuda.stream(h2d):
                    for hg, g in zip(host_g, sets[1 - b][0]):
                        g.copy_(hg, non_blocking=True)
                up[1 - b].record(h2d)
            compute.wait_event(up[b])
            if down[b] is not None:
                compute.wait_event(down[b])    # parameters of step i-2 downloaded
            if setup.w.get("master16") and down[1 - b] is not None:
                compute.wait_event(down[1 - b])  # one parameter buffer: step i-1's too
            sets[b][2](sp)
            done[b].record(compute)
            d2h.wait_event(done[b])
            with torch.cuda.stream(d2h):
                for hp_, p in zip(host_p, sets[b][1]):
                    hp_.copy_(p, non_blocking=True)
            down[b] = ev()
            down[b].record(d2h)
        compute.wait_stream(d2h)
        stop.record(compute)
        torch.cuda.synchronize()
        return start.elapsed_time(stop) / k

    run(2)
    return run(steps)


def link_rates(setup, reps=3):
    """GB/s of the step's own transfers with nothing else running: the
    gradients host->device alone, the 16-bit parameters device->host alone,
    and both at once on two streams (bytes of both / time), best of `reps`."""
    import torch
    host_g = [torch.empty(g.shape, dtype=g.dtype, pin_memory=True) for g in setup.grads]
    for hg, g in zip(host_g, setup.grads):
        hg.copy_(g)                       # the uploads write back the same gradients
    host_p = [torch.empty(p.shape, dtype=p.dtype, pin_memory=True) for p in setup.p16]
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()

    def timed(up, down):
        best = float("inf")
        for _ in range(reps):
            torch.cuda.synchronize()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            cur = torch.cuda.current_stream()
            a.record(cur)
            s1.wait_stream(cur)
            s2.wait_stream(cur)
            if up:
                with torch.cuda.stream(s1):
                    for hg, g in zip(host_g, setup.grads):
                        g.copy_(hg, non_blocking=True)
            if down:
                with torch.cuda.stream(s2):
                    for hp_, p in zip(host_p, setup.p16):
                        hp_.copy_(p, non_blocking=True)
            cur.wait_stream(s1)
            cur.wait_stream(s2)
            b.record(cur)
            torch.cuda.synchronize()
            best = min(best, a.elapsed_time(b) * 1e-3)
        return best

    bi, bo = setup.input_bytes(), setup.output_bytes()
    return {"h2d_gbs": bi / timed(True, False) / 1e9, "d2h_gbs": bo / timed(False, True) / 1e9,
            "both_gbs": (bi + bo) / timed(True, True) / 1e9}


def d2d_copy_gbs(dev, nbytes=1 << 30, reps=5):
    """A large device-to-device copy (cudaMemcpyAsync through torch), read +
    write bytes / time, best of `reps`: the achievable copy ceiling."""
    import torch
    a = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    b = torch.empty_like(a)
    best = float("inf")
    for _ in range(reps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        b.copy_(a)
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1) * 1e-3)
    del a, b
    return 2 * nbytes / best / 1e9


def run_ours(args):
    import torch
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    import __graft_entry__
    if rank == 0 or ws == 1:
        __graft_entry__.build()
    if ws > 1:
        torch.distributed.barrier()
        __graft_entry__.build()
    import zero_sharded_mixed_05_gb300 as z

    setup = Setup(args.workload, dev)
    w = setup.w
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    for _ in range(args.warmup):
        setup.step(sp)
    torch.cuda.synchronize()

    # per-pass events on the launching stream, for every timed step
    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    for trio in evs:
        for e in trio:
            e.record(stream)   # every event has a recorded state before the region
    torch.cuda.synchronize()
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    # keep the GPU busy while the sampler starts
    t_spin = time.time()
    while time.time() - t_spin < 0.3:
        setup.step(sp)
    launches0 = z.zero_opt_launch_count(setup.h)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    # Per-pass CUDA events (the timing hook) on every EVERY-th timed step.  An
    # event recorded between the two passes turns pass 2's programmatic
    # dependent launch into an ordinary one, so the other steps run exactly
    # as a caller runs them.
    EVERY = 8
    sampled = list(range(0, K, EVERY))
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    start.record(stream)
    for i in range(K):
        if i % EVERY == 0:
            z.zero_opt_set_events(setup.h, *evs[i])
            setup.step(sp)
            z.zero_opt_set_events(setup.h)
        else:
            setup.step(sp)
    end.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    launches = z.zero_opt_launch_count(setup.h) - launches0
    if ws > 1:
        torch.distributed.barrier()
    ms_total = start.elapsed_time(end)
    # keep sampling a little after the region, then stop
    clocks.stop()
    clk = clocks.summary(t0, t1)
    p1 = [evs[i][0].elapsed_time(evs[i][1]) for i in sampled]
    p2 = [evs[i][1].elapsed_time(evs[i][2]) for i in sampled]
    if ws > 1:
        ms_total = max_over_ranks(ms_total, dev)
    ms_step = ms_total / K
    n = setup.n
    value = ws * n / (ms_step * 1e-3)
    peak, peak_src = load_peaks()
    step_bytes = algorithmic_bytes_per_param(w) * n
    stash = setup.stash is not None
    p2_bytes = pass2_bytes_per_param(w, stash) * n
    p2_ms = statistics.mean(p2)
    p1_ms = statistics.mean(p1)
    achieved = p2_bytes / (p2_ms * 1e-3) / 1e9
    step_gbs = step_bytes / (ms_step * 1e-3) / 1e9

    # End to end through the public API with host buffers: every step's
    # gradients come from pinned host memory (H2D) and its 16-bit parameters
    # go back to pinned host memory (D2H), inside the timed region.  As in a
    # training loop, transfers overlap compute: the upload of step i+1's
    # gradients (into a second device buffer set) and the download of step
    # i's parameters (from one of two alternating parameter buffers) run on
    # their own streams while step i+1 computes.
    # The host side of the machine is shared, so the link-bound figure varies from
    # run to run: the median of three repetitions is reported, with all three.
    e2e = None
    if not args.no_e2e:
        e2e_runs = [e2e_pipelined(setup, stream, max(3, min(K, 50))) for _ in range(3)]
        e2e_ms = statistics.median(e2e_runs)
        if ws > 1:
            e2e_ms = max_over_ranks(e2e_ms, dev)
        e2e = {"value": ws * n / (e2e_ms * 1e-3), "unit": "params/s",
               "h2d_bytes_per_step": setup.input_bytes(),
               "d2h_bytes_per_step": setup.output_bytes(), "ms_per_step": e2e_ms,
               "ms_per_step_runs": e2e_runs,
               "transfers": "pinned host buffers; H2D and D2H on their own streams, "
                            "double-buffered device copies, overlapped with the steps; "
                            "median of 3 repetitions",
               "link_gbs": link_rates(setup)}
    d2d = d2d_copy_gbs(dev) if not args.no_e2e else None

    tpp, tsrc = pass2_traffic_per_param(args.workload) if not stash else (None, None)
    if w.get("div", 1) != 1 or args.numel:
        tpp = None                    # a resized workload has no committed capture
    traffic = tpp * n if tpp is not None else None
    traffic_src = ("ncu dram__bytes_read.sum + dram__bytes_write.sum of one pass-2 launch, "
                   "per parameter, times this workload's parameters (%s)" % tsrc
                   if traffic is not None else None)

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        sample = OracleSample(args.workload)
        rate = sample.rate(args.cpu_seconds)
        cpu = {"value": rate, "unit": "params/s", **sample.info()}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "params/s", "n_gpus": ws, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded SplitMix64 / Irwin-Hall), resident in HBM",
            "config": {"workload": w["desc"], "params_per_gpu": n,
                       "grad_dtype": w["dtype"], "grad_buffers": w["R"] * w["K"],
                       "l2": "inputs larger than L2 (algorithmic %.2f GB per step)" % (step_bytes / 1e9),
                       "stash": stash},
            "hbm_gbs": step_gbs, "hbm_frac": step_gbs / peak,
            "d2d_copy_gbs": d2d,
            "algorithmic_bytes_per_param": algorithmic_bytes_per_param(w),
            "roofline": {"bound": "hbm", "kernel": "pass2_kernel (unscale+clip+AdamW+cast)",
                         "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_source": peak_src + " (hbm_gbs)",
                         "traffic": traffic, "traffic_source": traffic_src,
                         "bytes_per_launch": p2_bytes,
                         "avg_launch_ms": p2_ms, "pass1_avg_ms": p1_ms,
                         "launches_timed": len(sampled),
                         "timing": "CUDA events around each pass on every %d-th timed "
                                   "step" % EVERY},
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": clk,
        }
        if cpu is not None:
            line["cpu_baseline"] = cpu
    if ws > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        emit(line)
    return 0


def run_sharded(args, stage):
    """The ZeRO-2 (stage 2) or ZeRO-3 (stage 3) data-parallel step of the
    workload's whole model sharded over the process group's N ranks (strong
    scaling: the model is fixed, each rank owns S = ceil(Psi / N) parameters).
    Every rank holds its local gradients for the whole model (K buffers of P
    elements), sends each shard's bytes to its owner (all-to-all), the owner
    folds the N ranks' statistics on the device and steps its shard, and under
    ZeRO-2 the 16-bit parameters are all-gathered.  The per-tensor list is
    taken as its flat concatenation (2,270,232,576 parameters), as a ZeRO
    engine keeps its gradients in contiguous buffers.  Prints one JSON line
    with the whole model's params/s."""
    import torch
    import torch.distributed as dist

    import synth
    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    os.environ.setdefault("MASTER_PORT", "29511")
    os.environ.setdefault("NCCL_NVLS_ENABLE", "0")
    dist.init_process_group("nccl", rank=rank, world_size=ws, device_id=dev)
    import __graft_entry__
    if rank == 0:
        __graft_entry__.build()
    dist.barrier()
    __graft_entry__.build()
    import zero_sharded_mixed_05_gb300 as z
    from zero_sharded_mixed_05_gb300.distributed import ZeroStep
    w = WORKLOADS[args.workload]
    psi, K = w["numel"], w["K"]           # the process group's ranks replace R
    code = z.FP16 if w["dtype"] == "fp16" else z.BF16
    kind = synth.F16 if code == z.FP16 else synth.BF16
    tdt = torch.float16 if code == z.FP16 else torch.bfloat16
    cfg = z.make_config(numel=psi, world=ws, grad_dtype=code, lr=w["lr"], weight_decay=w["wd"],
                        max_grad_norm=w["clip"], dynamic_scale=w["dynamic"],
                        init_scale=w["scale"], scale_window=1000,
                        master16=w.get("master16", False))
    zs = ZeroStep(cfg, backend="device", stage=stage)
    S, P = zs.S, zs.P
    b0, e0 = rank * S, min(psi, (rank + 1) * S)
    master = torch.zeros(S, dtype=torch.float32, device=dev)
    if e0 > b0:
        synth.fill_gpu(master[:e0 - b0], w["seed"], 0, b0, 0.02, synth.F32)
    m, v = torch.zeros(S, device=dev), torch.zeros(S, device=dev)
    if stage == 2:
        p16 = torch.zeros(P, dtype=tdt, device=dev)
        p16[b0:b0 + S].copy_(master)
        own16 = p16[b0:b0 + S]
    else:
        p16 = master.to(tdt)
        own16 = p16
    if w.get("master16"):
        master = None
    grads = []
    for k in range(K):
        g = torch.zeros(P, dtype=tdt, device=dev)
        synth.fill_gpu(g[:psi], w["seed"], 1 + rank * K + k, 0, w["sigma"] * w["scale"], kind)
        grads.append(g)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        zs.step(grads, master, m, v, p16)
    torch.cuda.synchronize()
    dist.barrier()
    EVERY = 8
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)]
           for _ in range(0, args.steps, EVERY)]
    for trio in evs:
        for e in trio:
            e.record(stream)   # torch times only events it has recorded once
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    t_spin = time.time()
    while time.time() - t_spin < 0.3:
        zs.step(grads, master, m, v, p16)
    launches0 = z.zero_opt_launch_count(zs.h)
    torch.cuda.synchronize()
    dist.barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    a.record(stream)
    for i in range(args.steps):
        if i % EVERY == 0:
            z.zero_opt_set_events(zs.h, *evs[i // EVERY])
            zs.step(grads, master, m, v, p16)
            z.zero_opt_set_events(zs.h)
        else:
            zs.step(grads, master, m, v, p16)
    b.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    launches = z.zero_opt_launch_count(zs.h) - launches0
    dist.barrier()
    clocks.stop()
    clk = clocks.summary(t0, t1)
    ms = max_over_ranks(a.elapsed_time(b) / args.steps, dev)
    p2_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    p2_ms = max_over_ranks(p2_ms, dev)
    nbuf = ws * K
    p2_bytes = (2 * nbuf + state_bytes_per_param(w)) * S
    peak, peak_src = load_peaks()
    # end to end: each step's local gradients come up from pinned host memory
    # and the rank's updated 16-bit shard goes back down, on the step's stream
    host_g = [torch.empty(g.shape, dtype=g.dtype, pin_memory=True) for g in grads]
    for hg, g in zip(host_g, grads):
        hg.copy_(g)
    host_p = torch.empty(own16.shape, dtype=own16.dtype, pin_memory=True)
    ke = max(3, min(args.steps, 20))
    torch.cuda.synchronize()
    dist.barrier()
    ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ea.record(stream)
    for _ in range(ke):
        for hg, g in zip(host_g, grads):
            g.copy_(hg, non_blocking=True)
        zs.step(grads, master, m, v, p16)
        host_p.copy_(own16, non_blocking=True)
    eb.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(ea.elapsed_time(eb) / ke, dev)
    line = None
    if rank == 0:
        name = "ZeRO-2" if stage == 2 else "ZeRO-3"
        line = {
            "metric": METRIC, "value": psi / (ms * 1e-3), "unit": "params/s",
            "impl": "zero%d" % stage, "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "strong",
            "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded SplitMix64 / Irwin-Hall), resident in HBM",
            "config": {"workload": w["desc"] + f" [{name} across the {ws} ranks: all-to-all of "
                       "the gradient bytes, statistics folded on the device, step of the own "
                       "shard" + (", all-gather of the 16-bit parameters" if stage == 2 else
                                  "; 16-bit parameters stay sharded") + "]",
                       "params_total": psi, "params_per_gpu": S, "micro_steps": K,
                       "parallelism": f"zero{stage}-dp{ws}",
                       "l2": "inputs larger than L2"},
            "roofline": {"bound": "hbm", "kernel": "pass2_kernel (unscale+clip+AdamW+cast) "
                         f"over the {nbuf} received shard buffers",
                         "achieved": p2_bytes / (p2_ms * 1e-3) / 1e9, "peak": peak,
                         "unit": "GB/s", "frac": p2_bytes / (p2_ms * 1e-3) / 1e9 / peak,
                         "peak_source": peak_src + " (hbm_gbs)", "traffic": None,
                         "bytes_per_launch": p2_bytes, "avg_launch_ms": p2_ms,
                         "timing": "CUDA events around each pass on every %d-th timed "
                                   "step" % EVERY},
            "e2e": {"value": psi / (e2e_ms * 1e-3), "unit": "params/s",
                    "h2d_bytes_per_step": sum(g.numel() * 2 for g in grads),
                    "d2h_bytes_per_step": own16.numel() * 2, "ms_per_step": e2e_ms,
                    "transfers": "pinned host buffers, copies in line with the step on its "
                                 "stream (each rank's local gradients up, its 16-bit shard "
                                 "down)"},
            "gpu_launches": launches, "clocks": clk}
    zs.close()
    dist.destroy_process_group()
    if line is not None:
        emit(line)
    return 0


def run_offload(args):
    """The offloaded step (zero_host_step) of a flat workload on host buffers,
    run by CPU threads: params/s over `--steps` steps after `--warmup`."""
    import synth
    import zero_sharded_mixed_05_gb300 as z
    w = WORKLOADS[args.workload]
    if args.workload == "pertensor":
        raise SystemExit("--offload applies to flat workloads")
    code = z.FP16 if w["dtype"] == "fp16" else z.BF16
    kind = synth.F16 if code == z.FP16 else synth.BF16
    cfg = z.make_config(numel=w["numel"], world=w["world"], grad_dtype=code, lr=w["lr"],
                        weight_decay=w["wd"], max_grad_norm=w["clip"],
                        dynamic_scale=w["dynamic"], init_scale=w["scale"], scale_window=1000,
                        master16=w.get("master16", False))
    h = z.zero_host_create(cfg, args.threads)
    S = -(-w["numel"] // w["world"])
    b, n = 0, min(S, w["numel"])                     # rank 0's shard
    master = synth.normal_np(w["seed"], 0, b, n, 0.02, synth.F32)
    p16 = z_cast16(master, code)
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    nb = w["R"] * w["K"]
    grads = [synth.normal_np(w["seed"], 1 + i, b, n, w["sigma"] * w["scale"], kind)
             for i in range(nb)]
    bufs = z.make_buffers(None if w.get("master16") else master, m, v, p16, grads,
                          n_ranks=w["R"], n_micro=w["K"], grads_shard_local=True,
                          param16_shard_local=True)
    for _ in range(args.warmup):
        z.zero_host_step(h, 0, bufs)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        z.zero_host_step(h, 0, bufs)
    dt = (time.perf_counter() - t0) / args.steps
    threads = z.zero_host_threads(h)
    z.zero_host_destroy(h)
    print(json.dumps({
        "metric": "offloaded optimizer-step params/s (host threads, host-resident state)",
        "value": n / dt, "unit": "params/s", "impl": "offload", "threads": threads,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "dtype": "f32", "data": "synthetic",
        "host_gbs": algorithmic_bytes_per_param(w) * n / dt / 1e9,
        "config": {"workload": w["desc"], "params": n, "cpu": platform.machine()}}))


def z_cast16(x, code):
    """Host 16-bit copy (round to nearest even) of fp32 values, via torch."""
    import torch
    dt = torch.float16 if code == 0 else torch.bfloat16
    return torch.from_numpy(x).to(dt).view(torch.int16).numpy().view(np.uint16).copy()


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="pertensor")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--numel", type=int, default=0,
                    help="override the flat workload's parameters per shard (profiling runs)")
    ap.add_argument("--div", type=int, default=1,
                    help="divide every dimension of the per-tensor list by this (profiling runs)")
    ap.add_argument("--no-e2e", action="store_true",
                    help="leave out the end-to-end and copy-ceiling legs (profiling runs)")
    ap.add_argument("--zero2", action="store_true",
                    help="time the sharded ZeRO-2 step with its collectives over the process "
                         "group (the default under torchrun with more than one rank)")
    ap.add_argument("--zero3", action="store_true",
                    help="time the sharded ZeRO-3 step (16-bit parameters stay sharded)")
    ap.add_argument("--replicas", action="store_true",
                    help="under torchrun, time independent replicas of the one-GPU step "
                         "instead of the sharded step")
    ap.add_argument("--offload", action="store_true",
                    help="time the offloaded step (CPU threads, host buffers) instead")
    ap.add_argument("--threads", type=int, default=0,
                    help="threads of the offloaded step (0: all hardware threads)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.numel:
        if args.workload == "pertensor":
            ap.error("--numel applies to flat workloads")
        w = dict(WORKLOADS[args.workload])
        w["numel"] = args.numel * w["world"]
        w["desc"] = w["desc"] + f" [resized to {args.numel:,} params per shard]"
        WORKLOADS[args.workload] = w
    if args.div != 1:
        if args.workload != "pertensor" or args.div < 1:
            ap.error("--div applies to the per-tensor list and must be >= 1")
        w = dict(WORKLOADS["pertensor"])
        w["div"] = args.div
        w["numel"] = int(sum(np.prod(shp) for shp in llama_shapes(args.div)))
        w["desc"] = w["desc"] + f" [every dimension divided by {args.div}: {w['numel']:,} params]"
        WORKLOADS["pertensor"] = w
    if args.impl == "reference":
        return run_reference(args)
    if args.offload:
        return run_offload(args)
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if args.zero3:
        return run_sharded(args, 3)
    if args.zero2 or (ws > 1 and not args.replicas):
        return run_sharded(args, 2)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
