"""Run one operation of the training step on its own, at the shapes of a GPT-2 workload.

    python -m gpt_train_step_arena_b300.kernel_bench --op fc_fwd [--reps 20] [--workload gpt2_124m]

Ops: the matrix products of a layer (qkv_fwd, attproj_fwd, fc_fwd, fcproj_fwd,
lmhead_fwd, fc_dgrad, fc_wgrad, qkv_wgrad, lmhead_dgrad, lmhead_wgrad), attention
(attn_fwd, attn_bwd), the fused-epilogue products (fc_fwd_gelu, fcproj_dgrad_gelu,
attproj_fwd_res, qkv_fwd_bias), layernorm (ln_fwd, ln_bwd), softmax + cross-entropy (xent), bias
gradients (bias_grad, bias_grad_fc, bias_grad_qkv) and AdamW over the full parameter
count.  Inputs are seeded random
device tensors; each op runs --reps times after --warmup runs, timed with CUDA events,
and prints one JSON line (ms per run, TFLOP/s or GB/s).  Used for per-kernel timing and
as the small, self-contained program that Nsight Compute captures.
"""
from __future__ import annotations

import argparse
import json

import torch

from . import ops, synth


def _gemm_case(name, c):
    M, C, Vp = c["B"] * c["T"], c["C"], (c["V"] + 127) // 128 * 128
    shapes = {  # (M, N, K, layout)
        "qkv_fwd": (M, 3 * C, C, "fwd"), "attproj_fwd": (M, C, C, "fwd"), "fc_fwd": (M, 4 * C, C, "fwd"),
        "fcproj_fwd": (M, C, 4 * C, "fwd"), "lmhead_fwd": (M, Vp, C, "fwd"),
        "fc_dgrad": (M, C, 4 * C, "dgrad"), "fcproj_dgrad": (M, 4 * C, C, "dgrad"),
        "lmhead_dgrad": (M, C, Vp, "dgrad"),
        "fc_wgrad": (4 * C, C, M, "wgrad"), "qkv_wgrad": (3 * C, C, M, "wgrad"),
        "attproj_wgrad": (C, C, M, "wgrad"), "lmhead_wgrad": (Vp, C, M, "wgrad"),
    }
    return shapes[name]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--op", required=True)
    ap.add_argument("--workload", default="gpt2_124m")
    ap.add_argument("--batch", type=int, default=None, help="override B (smaller device footprint)")
    ap.add_argument("--reps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--tile-rows", type=int, default=0,
                    help="force the tensor-core GEMM's tiles: 128, 256 or 2 (two-SM pairs); 0: per shape")
    args = ap.parse_args()
    if args.tile_rows:
        from . import _native as N_
        N_.lib.gpt2_op_gemm_force_tile_rows(args.tile_rows)
    c = dict(synth.WORKLOADS[args.workload])
    if args.batch:
        c["B"] = args.batch
    dev = "cuda"
    g = torch.Generator(device=dev).manual_seed(0)
    bf = torch.bfloat16

    def rnd(*shape, dtype=bf):
        return (torch.randn(*shape, device=dev, generator=g) * 0.5).to(dtype)

    if args.op.startswith("attn"):
        B, T, C, NH = c["B"], c["T"], c["C"], c["NH"]
        qkv = rnd(B, T, 3 * C)
        out, lse = ops.attention_forward(qkv, NH)
        dout = rnd(B, T, C)
        flops = 2.0 * B * NH * (C // NH) * T * (T + 1)
        if args.op == "attn_fwd":
            fn = lambda: ops.attention_forward(qkv, NH)
        else:
            fn = lambda: ops.attention_backward(dout, qkv, out, lse, NH)
            flops *= 2
        unit, work = "TFLOP/s", flops
    elif args.op in ("ln_fwd", "ln_bwd"):
        M, C = c["B"] * c["T"], c["C"]
        x, dy, acc = rnd(M, C), rnd(M, C), rnd(M, C)
        w = torch.ones(C, device=dev) + 0.1 * torch.randn(C, device=dev, generator=g)
        b = 0.1 * torch.randn(C, device=dev, generator=g)
        _, mean, rstd = ops.layernorm_forward(x, w, b)
        if args.op == "ln_fwd":
            fn = lambda: ops.layernorm_forward(x, w, b)
            work = 2.0 * M * C * 2 + 8.0 * M
        else:
            fn = lambda: ops.layernorm_backward(acc, dy, x, w, mean, rstd)
            work = 4.0 * M * C * 2 + 8.0 * M
        unit = "GB/s"
    elif args.op == "xent":
        M, V = c["B"] * c["T"], c["V"]
        Vp = (V + 127) // 128 * 128
        logits = rnd(M, Vp)
        tg = torch.randint(0, V, (M,), device=dev, dtype=torch.int32, generator=g)
        fn = lambda: ops.softmax_xent(logits, tg, V, 1.0 / M, check=False)
        unit, work = "GB/s", 2.0 * M * Vp * 2 + 8.0 * M
    elif args.op.startswith("bias_grad"):
        M = c["B"] * c["T"]
        Nn = {"bias_grad": c["C"], "bias_grad_fc": 4 * c["C"], "bias_grad_qkv": 3 * c["C"]}[args.op]
        x = rnd(M, Nn)
        fn = lambda: ops.bias_grad(x)
        unit, work = "GB/s", 2.0 * M * Nn + 4.0 * Nn
    elif args.op == "adamw":
        n = sum(synth.param_sizes(c["L"], c["C"], (c["V"] + 127) // 128 * 128, c["maxT"]))
        p, gr, m, v = (rnd(n, dtype=torch.float32) for _ in range(4))
        v.abs_()
        sh = torch.empty(n, dtype=bf, device=dev)
        fn = lambda: ops.adamw(p, gr, m, v, 6e-4, 0.9, 0.999, 1e-8, 0.1, 1, shadow=sh)
        unit, work = "GB/s", 30.0 * n
    elif args.op in ("fc_fwd_gelu", "fcproj_dgrad_gelu", "attproj_fwd_res", "qkv_fwd_bias"):
        # the products with the epilogues the training step fuses into them
        from . import _native as N_
        M, C = c["B"] * c["T"], c["C"]
        bias = lambda n: 0.1 * torch.randn(n, device=dev, generator=g)
        if args.op == "fc_fwd_gelu":
            A, W, b = rnd(M, C), rnd(4 * C, C), bias(4 * C)
            fn = lambda: ops.linear_fused(A, W, N_.GPT2_EPI_GELU, bias=b)
            Nn, K = 4 * C, C
        elif args.op == "fcproj_dgrad_gelu":
            A, W, P = rnd(M, C), rnd(C, 4 * C), rnd(M, 4 * C)
            fn = lambda: ops.linear_fused(A, W, N_.GPT2_EPI_GELU_BWD, P=P, b_kmajor=False)
            Nn, K = 4 * C, C
        elif args.op == "attproj_fwd_res":
            A, W, b, R = rnd(M, C), rnd(C, C), bias(C), rnd(M, C)
            fn = lambda: ops.linear_fused(A, W, N_.GPT2_EPI_STORE, bias=b, R=R)
            Nn, K = C, C
        else:
            A, W, b = rnd(M, C), rnd(3 * C, C), bias(3 * C)
            fn = lambda: ops.linear_fused(A, W, N_.GPT2_EPI_STORE, bias=b)
            Nn, K = 3 * C, C
        unit, work = "TFLOP/s", 2.0 * M * Nn * K
    else:
        M, N, K, layout = _gemm_case(args.op, c)
        if layout == "fwd":
            A, Bm = rnd(M, K), rnd(N, K)
            fn = lambda: ops.matmul(A, Bm, True, True)
        elif layout == "dgrad":
            A, Bm = rnd(M, K), rnd(K, N)
            fn = lambda: ops.matmul(A, Bm, True, False)
        else:
            A, Bm = rnd(K, M), rnd(K, N)
            ws = 1 << 28
            fn = lambda: ops.matmul(A, Bm, False, False, out_f32=True, workspace_bytes=ws)
        unit, work = "TFLOP/s", 2.0 * M * N * K
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.reps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.reps
    rate = work / (ms / 1e3) / (1e12 if unit == "TFLOP/s" else 1e9)
    print(json.dumps({"op": args.op, "workload": args.workload, "B": c["B"], "ms": ms, unit: rate,
                      "variant": ops.gemm_last_variant()}))


if __name__ == "__main__":
    main()
