#!/usr/bin/env python3
"""Throughput of one GPT-2 training step (forward + backward + AdamW) on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload gpt2_124m|gpt2_350m|...] [--norm layernorm|rmsnorm]

Prints ONE JSON line on rank 0.  The workload is GPT-2 124M (L=12, C=768, H=12,
V=50257 padded to 50304 on the device) at B=32, T=1024 in bf16 mixed precision, on a
seeded synthetic Zipf(1.1) token stream with N(0, 0.02) initial weights.

`value` times W warm-up steps and then K steps with the ids already resident in device
memory (CUDA events on the library's stream, max over ranks).  `e2e` times K more steps
through the public host-pointer call gpt2_forward (ids copied from pinned host memory,
the loss read back every step).  With N > 1, each rank trains its own independent
replica on its own slice of the token stream (the step has no cross-rank exchange in
this build), so scaling is weak.

--norm rmsnorm runs the microGPT variant of the same shapes (every LayerNorm replaced
by RMSNorm, page "microGPT 3D", lesson 04).

--impl reference times the CPU oracle (test infrastructure, plain C, all host cores)
on bounded samples of the same workload, rank 0 only: fwd+bwd on B=1,T=--cpu-tokens
positions plus one AdamW over all parameters per step, extrapolated to the step's B*T
positions (workloads of at most 4096 tokens per step are timed in full).  The same
sample gives the `cpu_baseline` of the default arm; --cpu-variants adds the double and
float oracles on one thread and on every core.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "training tokens/sec (fwd+bwd+AdamW) for GPT-2 124M at B=32,T=1024; MFU vs BF16 peak"
DATA = "synthetic: seeded Zipf(s=1.1) token stream (xorshift64*), N(0,0.02) init"


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sus=d["bf16_tflops_sustained"],
                    source="measured")
    return dict(hbm=6400.0, bf16=1800.0, bf16_sus=1400.0, source="fallback")


def flops_per_token(c, Vp):
    """Algorithmic train FLOPs per token: GEMMs 6*(12*L*C^2 + Vp*C) plus causal attention
    3 * 2 * C * (T+1) * L (QK^T and PV over t2 <= t; backward = 2x forward)."""
    L, C, T = c["L"], c["C"], c["T"]
    return 6.0 * (12 * L * C * C + Vp * C) + 3.0 * 2.0 * C * (T + 1) * L


def palm_flops_per_token(c, Vp):
    """The PaLM-paper convention, reported beside the algorithmic count: 6 N + 12 L C T
    per token, N = every parameter (the padded wte included)."""
    from gpt_train_step_arena_b300 import synth
    n = sum(synth.param_sizes(c["L"], c["C"], Vp, c["maxT"]))
    return 6.0 * n + 12.0 * c["L"] * c["C"] * c["T"]


def measure_tf32_peak():
    """Dense TF32 matmul throughput of this GPU (TFLOP/s): torch fp32 8192^3 with TF32
    allowed, best of 10 after warm-up, CUDA events."""
    import torch
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = True
    n = 8192
    g = torch.Generator(device="cuda").manual_seed(0)
    a = torch.randn(n, n, device="cuda", generator=g)
    b = torch.randn(n, n, device="cuda", generator=g)
    for _ in range(3):
        torch.matmul(a, b)
    best = float("inf")
    for _ in range(10):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        torch.matmul(a, b)
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1))
    torch.backends.cuda.matmul.allow_tf32 = prev
    del a, b
    return 2.0 * n ** 3 / (best / 1e3) / 1e12


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.path = os.path.join("/tmp", f"bench_clocks_{os.getpid()}.csv")
        self.proc = None
        self.gpu = gpu_index

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "200"], stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons, power = [], None, set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.remove(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power) if power else None}


# ------------------------------------------------------------------ distributed
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ traffic from ncu
def recorded_traffic(kernel_class: str):
    """dram bytes per launch measured by ncu for this kernel class, if the summary under
    profiles/ was taken on the current source of that kernel (else None)."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(kernel_class)
    if not d:
        return None
    h = hashlib.sha256()
    for f in d.get("sources", []):
        fp = os.path.join(ROOT, f)
        if not os.path.exists(fp):
            return None
        h.update(open(fp, "rb").read())
    if h.hexdigest() != d.get("sha256"):
        return None
    return d.get("bytes_per_launch")


# ------------------------------------------------------------------ oracle (CPU) timing
def cpu_model() -> str:
    try:
        for line in open("/proc/cpuinfo"):
            if line.startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


FULL_STEP_TOKENS = 4096  # workloads up to this many tokens per step are timed in full


def sample_shape(cfg, cpu_tokens):
    """(B, T) of the oracle's CPU sample: the whole step for small workloads, else the
    first cpu_tokens positions of row 0 (B=1)."""
    if cfg["B"] * cfg["T"] <= FULL_STEP_TOKENS:
        return cfg["B"], cfg["T"]
    return 1, min(cpu_tokens, cfg["T"])


def oracle_sample(cfg, B_s, T_s, stream_seed=1337, norm="layernorm", variant="f64"):
    """The CPU oracle set up for one bounded sample of the workload: the full model on the
    first B_s x T_s positions of step 0 (B_s = 1: the first T_s positions of row 0)."""
    from gpt_train_step_arena_b300 import synth
    from oracle.oracle import Model, cpu_threads
    L, C, NH, V, maxT = cfg["L"], cfg["C"], cfg["NH"], cfg["V"], cfg["maxT"]
    params = synth.init_params(L, C, V, maxT, seed=42)
    stream = synth.token_stream(cfg, steps=1, seed=stream_seed)
    if B_s == 1:
        inp = stream[:T_s].reshape(1, T_s)
        tgt = stream[1:T_s + 1].reshape(1, T_s)
    else:
        assert T_s == cfg["T"], "a multi-row sample takes whole rows"
        inp, tgt = synth.batch(stream, 0, B_s, T_s)
    m = Model(L, C, NH, V, maxT, variant=variant, norm=norm)
    m.set_params(params)
    return m, inp, tgt, cpu_threads()


def oracle_step_time(m, inp, tgt, hp, t):
    """(fwd+bwd seconds on the sample, AdamW seconds over all parameters) of one step."""
    t0 = time.perf_counter()
    m.forward(inp, tgt)
    m.backward()
    t1 = time.perf_counter()
    m.update(*hp, t)
    return t1 - t0, time.perf_counter() - t1


def extrapolated_tokens_per_s(cfg, sample_tokens, t_fb, t_adam):
    """Tokens/s of the full step from the sample: the step's B*T positions cost
    B*T/sample_tokens times the sample's fwd+bwd, plus one AdamW over all parameters
    (exact when the sample is the whole step)."""
    BT = cfg["B"] * cfg["T"]
    return BT / (BT / sample_tokens * t_fb + t_adam)


def cpu_sample_text(workload, B_s, T_s, t_fb, t_adam, variant="f64", threads="OpenMP on the host cores"):
    if B_s > 1:
        return (f"full step: fwd+bwd of the {workload} model on its B={B_s},T={T_s} batch of step 0 "
                f"({t_fb:.3g} s) plus one AdamW over all parameters ({t_adam:.3g} s); {variant} oracle, {threads}")
    return (f"extrapolated: fwd+bwd of the full {workload} model on B=1,T={T_s} (the first {T_s} positions of "
            f"row 0 of step 0; {t_fb:.3g} s) scaled to the step's B*T positions, plus one AdamW over all "
            f"parameters ({t_adam:.3g} s); {variant} oracle, {threads}. Per-token attention work "
            f"grows with T, so at T=1024 the oracle's step costs a few percent more per token than this")


def cpu_leg(cfg, workload, norm, cpu_tokens, hp, t=1, variant="f64", threads=0):
    """The oracle timed on one sample step: (tokens/s of the whole step, threads used, sample text).
    threads: 0 = the OpenMP default (the cores this process may run on, or OMP_NUM_THREADS),
    else that many."""
    from oracle.oracle import set_threads
    B_s, T_s = sample_shape(cfg, cpu_tokens)
    m, inp, tgt, _ = oracle_sample(cfg, B_s, T_s, norm=norm, variant=variant)
    prev = set_threads(0, variant)
    used = set_threads(threads, variant) if threads > 0 else prev
    try:
        t_fb, t_adam = oracle_step_time(m, inp, tgt, hp, t)
    finally:
        set_threads(prev, variant)
    del m
    text = cpu_sample_text(workload, B_s, T_s, t_fb, t_adam, variant,
                           "one thread" if used == 1 else f"OpenMP, {used} threads")
    return extrapolated_tokens_per_s(cfg, B_s * T_s, t_fb, t_adam), used, text


def cpu_variants(cfg, workload, norm, cpu_tokens, hp):
    """The double and float oracles, each on one thread and on every host core, on the same
    sample (one step each, after one untimed step)."""
    out = []
    for variant in ("f64", "f32"):
        for threads in (1, 0):
            cpu_leg(cfg, workload, norm, cpu_tokens, hp, 1, variant, threads)   # untimed: page in, warm caches
            v, used, text = cpu_leg(cfg, workload, norm, cpu_tokens, hp, 2, variant, threads)
            out.append({"oracle": variant, "threads": used, "value": v, "unit": "tokens/s", "sample": text})
    return out


def cpu_host_info():
    return {"cpu_model": cpu_model(), "nproc": os.cpu_count(),
            "OMP_NUM_THREADS": os.environ.get("OMP_NUM_THREADS")}


def run_reference(args, rank, world):
    """--impl reference: the oracle on the host cores, rank 0 only."""
    if rank != 0:
        return
    from gpt_train_step_arena_b300 import synth
    cfg = dict(synth.WORKLOADS[args.workload])
    B_s, T_s = sample_shape(cfg, args.cpu_tokens)
    m, inp, tgt, cores = oracle_sample(cfg, B_s, T_s, norm=args.norm)
    hp = (cfg["lr"], cfg["b1"], cfg["b2"], cfg["eps"], cfg["wd"])
    for i in range(args.warmup):
        oracle_step_time(m, inp, tgt, hp, i + 1)
    t_fb = t_adam = 0.0
    for i in range(args.steps):
        a, b = oracle_step_time(m, inp, tgt, hp, args.warmup + i + 1)
        t_fb += a
        t_adam += b
    t_fb /= args.steps
    t_adam /= args.steps
    value = extrapolated_tokens_per_s(cfg, B_s * T_s, t_fb, t_adam)
    sample = cpu_sample_text(args.workload, B_s, T_s, t_fb, t_adam)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000 * cfg["B"] * cfg["T"] / value,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": DATA, "config": config_block(cfg, args.workload, args.norm),
        "cpu_baseline": dict({"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                              "sample": sample}, **cpu_host_info()),
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    if args.cpu_variants:
        del m
        line["cpu_variants"] = cpu_variants(cfg, args.workload, args.norm, args.cpu_tokens, hp)
    print(json.dumps(line), flush=True)


PRECISION_TEXT = {"bf16": "bf16 mixed (fp32 master/AdamW)", "tf32": "fp32 tensors, TF32 tensor-core matmuls",
                  "fp32": "strict fp32"}


def config_block(cfg, workload, norm="layernorm", precision="bf16"):
    Vp = (cfg["V"] + 127) // 128 * 128
    if norm != "layernorm":
        workload = f"{workload}_{norm}"   # the microGPT variant of the same shapes
    if precision != "bf16":
        workload = f"{workload}_{precision}"
    return {"workload": workload, "norm": norm, "L": cfg["L"], "C": cfg["C"], "H": cfg["NH"], "V": cfg["V"], "Vp": Vp,
            "B": cfg["B"], "T": cfg["T"], "precision": PRECISION_TEXT[precision],
            "lr": cfg["lr"], "wd": cfg["wd"],
            "l2": "no flush: every step streams > 10 GB of activations and weights, far above the 126 MB L2"}


# ------------------------------------------------------------------ our arm
def run_ours(args, rank, world, local):
    import numpy as np
    import torch
    from gpt_train_step_arena_b300 import synth
    from gpt_train_step_arena_b300.model import GPT2

    torch.cuda.set_device(local)
    cfg = dict(synth.WORKLOADS[args.workload])
    L, C, NH, V, maxT, B, T = (cfg[k] for k in ("L", "C", "NH", "V", "maxT", "B", "T"))
    hp = (cfg["lr"], cfg["b1"], cfg["b2"], cfg["eps"], cfg["wd"])
    W, K = args.warmup, args.steps
    params = synth.init_params(L, C, V, maxT, seed=42)
    stream = synth.token_stream(cfg, steps=W + 2 * K, seed=1337 + rank)
    batches = [synth.batch(stream, s, B, T) for s in range(W + 2 * K)]

    g = GPT2(L, C, NH, V, maxT, precision=args.precision, norm=args.norm)
    g.set_params(params)
    s = torch.cuda.Stream()
    g.set_stream(s.cuda_stream)
    tok_dev = torch.from_numpy(np.stack([b[0] for b in batches])).to(f"cuda:{local}")
    tgt_dev = torch.from_numpy(np.stack([b[1] for b in batches])).to(f"cuda:{local}")
    torch.cuda.synchronize()

    step_no = 0

    def dev_step(i):
        nonlocal step_no
        step_no += 1
        g.forward_async(tok_dev[i], tgt_dev[i], B, T, device=True)
        g.backward()
        g.update(*hp, step_no)

    for i in range(W):
        dev_step(i)
    first_loss = g.read_loss()
    torch.cuda.synchronize()
    barrier(world)

    # the timed region: no per-op instrumentation
    clocks = ClockSampler(local)
    clocks.start()
    launches0 = g.kernel_launches()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier(world)
    ev0.record(s)
    for i in range(W, W + K):
        dev_step(i)
    ev1.record(s)
    torch.cuda.synchronize()
    launches = g.kernel_launches() - launches0
    elapsed_ms = ev0.elapsed_time(ev1)
    clk = clocks.stop()
    last_loss = g.read_loss()
    barrier(world)
    max_ms = max_over_ranks(elapsed_ms, world)

    # a separate pass over the same batches with an event pair around every op, for the
    # per-class kernel times and the roofline entry
    g.profile_reset()
    g.profile_enable(True)
    for i in range(W, W + K):
        dev_step(i)
    torch.cuda.synchronize()
    g.profile_enable(False)
    prof = g.profile_read()

    # e2e: the public host-pointer call, ids from pinned host memory, loss read back
    tok_h = torch.from_numpy(np.stack([b[0] for b in batches])).pin_memory()
    tgt_h = torch.from_numpy(np.stack([b[1] for b in batches])).pin_memory()
    from gpt_train_step_arena_b300 import _native as N
    for i in range(W + K, W + K + 2):
        loss = N.lib.gpt2_forward(g.h, tok_h[i].data_ptr(), tgt_h[i].data_ptr(), B, T)
        g.backward()
        step_no += 1
        g.update(*hp, step_no)
    torch.cuda.synchronize()
    barrier(world)
    clocks_e2e = ClockSampler(local)
    clocks_e2e.start()
    t0 = time.perf_counter()
    for i in range(W + K, W + 2 * K):
        loss = N.lib.gpt2_forward(g.h, tok_h[i].data_ptr(), tgt_h[i].data_ptr(), B, T)
        if not math.isfinite(loss):
            raise RuntimeError(f"e2e forward failed: {N.lib.gpt2_last_error(g.h).decode()}")
        g.backward()
        step_no += 1
        g.update(*hp, step_no)
    g.sync()
    e2e_s = time.perf_counter() - t0
    clk_e2e = clocks_e2e.stop()
    e2e_s = max_over_ranks(e2e_s, world)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v_cpu, cores, text = cpu_leg(cfg, args.workload, args.norm, args.cpu_tokens, hp)
        cpu = dict({"value": v_cpu, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": text},
                   **cpu_host_info())
    cpu_var = None
    if rank == 0 and world == 1 and args.cpu_variants:
        cpu_var = cpu_variants(cfg, args.workload, args.norm, args.cpu_tokens, hp)

    tf32_peak = measure_tf32_peak() if args.precision == "tf32" and rank == 0 else None
    if rank != 0:
        return
    pk = _peaks()
    Vp = g.Vp
    fpt = flops_per_token(cfg, Vp)
    palm = palm_flops_per_token(cfg, Vp)
    ms_step = max_ms / K
    tokens = world * K * B * T
    value = tokens / (max_ms / 1000.0)
    kernels = {}
    for name, (ms, work, calls) in prof.items():
        if calls == 0:
            continue
        is_flops = name in ("gemm", "attn_fwd", "attn_bwd")
        kernels[name] = {"ms_per_step": ms / K, "calls_per_step": calls / K,
                         ("tflops" if is_flops else "gbs"): (work / (ms / 1e3)) / (1e12 if is_flops else 1e9)}
    dom = max(prof.items(), key=lambda kv: kv[1][0])
    dname, (dms, dwork, dcalls) = dom
    tensor = dname in ("gemm", "attn_fwd", "attn_bwd")
    if tensor:
        achieved = dwork / (dms / 1e3) / 1e12
        peak = pk["bf16_sus"]
        unit = "TFLOP/s"
    else:
        achieved = dwork / (dms / 1e3) / 1e9
        peak = pk["hbm"]
        unit = "GB/s"
    roofline = {"bound": "tensor" if tensor else "hbm", "kernel": dname, "achieved": achieved, "peak": peak,
                "unit": unit, "frac": achieved / peak, "traffic": recorded_traffic(dname),
                "peak_source": f"{pk['source']} ({'bf16 sustained' if tensor else 'HBM copy'})",
                "work_per_launch": dwork / dcalls, "ms_per_launch": dms / dcalls}
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": args.precision, "data": DATA, "config": config_block(cfg, args.workload, args.norm, args.precision),
        "mfu": ({"algorithmic_flops_per_token": fpt,
                 "vs_measured_burst": value / world * fpt / (pk["bf16"] * 1e12),
                 "vs_measured_sustained": value / world * fpt / (pk["bf16_sus"] * 1e12),
                 "palm_flops_per_token": palm,
                 "palm_vs_measured_burst": value / world * palm / (pk["bf16"] * 1e12),
                 "peak": "the 40% target is judged against the measured dense bf16 burst peak (cuBLAS, "
                         "MEASURED_PEAKS.json), the larger of the two measured figures"}
                if args.precision == "bf16" else
                {"algorithmic_flops_per_token": fpt,
                 "tf32_peak_tflops": tf32_peak,
                 "vs_tf32_peak": (value / world * fpt / (tf32_peak * 1e12)) if tf32_peak else None,
                 "peak": "dense TF32 peak measured in this run (cuBLAS fp32 8192^3 with TF32 allowed, best of 10)"}),
        "roofline": roofline,
        "kernels": kernels,
        "cpu_baseline": cpu,
        **({"cpu_variants": cpu_var} if cpu_var else {}),
        "e2e": {"value": world * K * B * T / e2e_s, "unit": "tokens/s",
                "h2d_bytes_per_step": 2 * B * T * 4, "d2h_bytes_per_step": 8, "clocks": clk_e2e},
        "gpu_launches": launches,
        "clocks": clk,
        "loss": {"after_warmup": first_loss, "last": last_loss},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ generation
GEN_METRIC = "generated tokens/sec (greedy decode with a key/value cache) for GPT-2 124M"


def gen_bytes_per_step(cfg, Vp, B, t):
    """Algorithmic HBM bytes of one one-token decode step at cache length t (positions
    0..t): every bf16 weight once (the 12*L*C^2 block matrices and the Vp*C tied head),
    plus the cached keys and values of B sequences read once, plus the new row's
    key/value written."""
    L, C = cfg["L"], cfg["C"]
    weights = 2 * (12 * L * C * C + Vp * C)
    kv = 2 * L * B * (t + 1) * 2 * C
    return weights + kv


def run_generate(args, rank, world, local):
    import numpy as np
    import torch
    from gpt_train_step_arena_b300 import synth
    from gpt_train_step_arena_b300.model import GPT2

    torch.cuda.set_device(local)
    cfg = dict(synth.WORKLOADS[args.workload])
    L, C, NH, V, maxT = (cfg[k] for k in ("L", "C", "NH", "V", "maxT"))
    B, T0, n_new = args.gen_batch, args.gen_prompt, args.gen_tokens
    params = synth.init_params(L, C, V, maxT, seed=42)
    stream = synth.token_stream(cfg, steps=1, seed=1337 + rank)
    prompt = stream[:B * T0].reshape(B, T0).astype(np.int32)
    g = GPT2(L, C, NH, V, maxT, precision="bf16", norm=args.norm)
    g.set_params(params)
    s = torch.cuda.Stream()
    g.set_stream(s.cuda_stream)
    for _ in range(args.warmup):
        g.generate(prompt, n_new)
    # the prompt pass alone, to separate it from the decode steps
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    ev[0].record(s)
    for _ in range(args.steps):
        g.generate(prompt, 1)
    ev[1].record(s)
    clocks = ClockSampler(local)
    clocks.start()
    launches0 = g.kernel_launches()
    barrier(world)
    t_host = time.perf_counter()
    ev[2].record(s)
    for _ in range(args.steps):
        out = g.generate(prompt, n_new)
    ev[3].record(s)
    torch.cuda.synchronize()
    t_host = time.perf_counter() - t_host
    clk = clocks.stop()
    launches = g.kernel_launches() - launches0
    prefill_ms = ev[0].elapsed_time(ev[1]) / args.steps
    total_ms = max_over_ranks(ev[2].elapsed_time(ev[3]) / args.steps, world)
    decode_ms = (total_ms - prefill_ms) / max(1, n_new - 1)
    if rank != 0:
        return
    pk = _peaks()
    Vp = g.Vp
    t_mid = T0 + (n_new - 1) // 2
    bytes_step = gen_bytes_per_step(cfg, Vp, B, t_mid)
    achieved = bytes_step / (decode_ms / 1e3) / 1e9
    value = world * B * n_new / (total_ms / 1e3)
    line = {
        "mode": "generate", "metric": GEN_METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": DATA,
        "config": {"workload": f"{args.workload}_generate" + ("" if args.norm == "layernorm" else f"_{args.norm}"),
                   "B": B, "prompt": T0, "new_tokens": n_new, "sampling": "greedy",
                   "step": "one gpt2_generate call: prompt pass + (new_tokens - 1) one-token decode steps",
                   "l2": "no flush: every decode step streams the 0.25 GB of bf16 weights, twice the L2"},
        "prefill_ms": prefill_ms, "decode_ms_per_token": decode_ms,
        "roofline": {"bound": "hbm", "kernel": "decode step (all kernels)", "achieved": achieved,
                     "peak": pk["hbm"], "unit": "GB/s", "frac": achieved / pk["hbm"], "traffic": None,
                     "peak_source": f"{pk['source']} (HBM copy)", "bytes_per_decode_step": bytes_step},
        "e2e": {"value": world * B * n_new / (t_host / args.steps), "unit": "tokens/s",
                "h2d_bytes_per_step": B * T0 * 4, "d2h_bytes_per_step": B * n_new * 4},
        "gpu_launches": launches,
        "clocks": clk,
        "sample_ids": out[0, :8].tolist(),
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ forward only
FWD_METRIC = "forward-only tokens/sec (logits of every position, no targets)"


def run_forward(args, rank, world, local):
    """The forward pass without targets (logits of every position, no loss): the
    inference half of the step, 1/3 of its algorithmic FLOPs."""
    import numpy as np
    import torch
    from gpt_train_step_arena_b300 import synth
    from gpt_train_step_arena_b300.model import GPT2

    torch.cuda.set_device(local)
    cfg = dict(synth.WORKLOADS[args.workload])
    L, C, NH, V, maxT, T = (cfg[k] for k in ("L", "C", "NH", "V", "maxT", "T"))
    B = args.fwd_batch or cfg["B"]
    W, K = args.warmup, args.steps
    params = synth.init_params(L, C, V, maxT, seed=42)
    stream = synth.token_stream(dict(cfg, B=B), steps=W + K, seed=1337 + rank)
    tok = np.stack([synth.batch(stream, i, B, T)[0] for i in range(W + K)])
    g = GPT2(L, C, NH, V, maxT, precision="bf16", norm=args.norm)
    g.set_params(params)
    s = torch.cuda.Stream()
    g.set_stream(s.cuda_stream)
    tok_dev = torch.from_numpy(tok).to(f"cuda:{local}")
    for i in range(W):
        g.forward_async(tok_dev[i], None, B, T, device=True)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    launches0 = g.kernel_launches()
    barrier(world)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(s)
    for i in range(W, W + K):
        g.forward_async(tok_dev[i], None, B, T, device=True)
    ev1.record(s)
    torch.cuda.synchronize()
    clk = clocks.stop()
    launches = g.kernel_launches() - launches0
    ms = max_over_ranks(ev0.elapsed_time(ev1) / K, world)
    # e2e: the public host-pointer call with ids from pinned host memory
    tok_h = torch.from_numpy(tok).pin_memory()
    from gpt_train_step_arena_b300 import _native as N
    t0 = time.perf_counter()
    for i in range(W, W + K):
        N.lib.gpt2_forward(g.h, tok_h[i].data_ptr(), None, B, T)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks((time.perf_counter() - t0) / K, world)
    if rank != 0:
        return
    pk = _peaks()
    fpt = flops_per_token(cfg, g.Vp) / 3.0
    value = world * B * T / (ms / 1e3)
    line = {
        "mode": "forward", "metric": FWD_METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": DATA,
        "config": dict(config_block(cfg, args.workload, args.norm), B=B, workload=f"{args.workload}_forward_b{B}"),
        "mfu": {"algorithmic_flops_per_token": fpt, "vs_measured_burst": value / world * fpt / (pk["bf16"] * 1e12)},
        "e2e": {"value": world * B * T / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": B * T * 4,
                "d2h_bytes_per_step": 0},
        "gpu_launches": launches,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="gpt2_124m")
    ap.add_argument("--mode", choices=["train", "generate", "forward"], default="train",
                    help="generate: greedy decode throughput with the key/value cache; "
                         "forward: logits of every position without targets")
    ap.add_argument("--fwd-batch", type=int, default=0, help="forward mode batch (default: the workload's B)")
    ap.add_argument("--gen-batch", type=int, default=16)
    ap.add_argument("--gen-prompt", type=int, default=64)
    ap.add_argument("--gen-tokens", type=int, default=40)
    ap.add_argument("--norm", choices=["layernorm", "rmsnorm"], default="layernorm",
                    help="rmsnorm: the microGPT variant (every LayerNorm replaced by RMSNorm)")
    ap.add_argument("--precision", choices=["bf16", "tf32", "fp32"], default="bf16",
                    help="train mode: tf32 = fp32 tensors with TF32 tensor-core matmuls (MFU against a TF32 peak "
                         "measured in the same run)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-tokens", type=int, default=128,
                    help="positions of the oracle's CPU sample (both arms), B=1, for workloads of more than "
                         f"{FULL_STEP_TOKENS} tokens per step (smaller ones are timed in full)")
    ap.add_argument("--cpu-variants", action="store_true",
                    help="also time the double and float oracles on one thread and on every host core "
                         "(cpu_variants; minutes at the 124M shapes)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, rank, world)
    elif args.mode == "generate":
        run_generate(args, rank, world, local)
    elif args.mode == "forward":
        run_forward(args, rank, world, local)
    else:
        run_ours(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
