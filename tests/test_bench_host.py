"""CPU checks of bench.py's host arithmetic: the algorithmic FLOPs per token behind the
MFU figure (recounted here layer by layer), the bytes of a one-token generation step,
and the JSON config block."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from gpt_train_step_arena_b300 import synth  # noqa: E402


def _recount(c, Vp):
    """Forward FLOPs per token, op by op, times 3 (backward = 2 x forward)."""
    L, C, T = c["L"], c["C"], c["T"]
    per_layer = 2 * C * 3 * C + 2 * C * C + 2 * C * 4 * C + 2 * 4 * C * C  # qkv, attproj, fc, fcproj
    head = 2 * C * Vp                                                     # tied LM head
    # causal attention: token t attends to t+1 keys; QK^T and PV are 2*hs FLOPs per key per
    # head each, i.e. 4*C per key; averaged over t = 0..T-1 that is 4*C*(T+1)/2 per token
    attn = 4 * C * (T + 1) / 2
    return 3 * (L * (per_layer + attn) + head)


def test_flops_per_token_matches_op_by_op_count():
    for name, want in (("gpt2_124m", 798_087_168), ("gpt2_350m", 2_272_149_504)):
        c = synth.WORKLOADS[name]
        Vp = (c["V"] + 127) // 128 * 128
        assert Vp == 50304
        got = bench.flops_per_token(c, Vp)
        assert got == _recount(c, Vp) == want, (name, got)
    # 26.15 TFLOP per 124M step of 32 x 1024 tokens
    c = synth.WORKLOADS["gpt2_124m"]
    assert abs(bench.flops_per_token(c, 50304) * 32 * 1024 / 1e12 - 26.152) < 1e-3


def test_generation_step_bytes():
    c = synth.WORKLOADS["gpt2_124m"]
    weights = 2 * (12 * 12 * 768 * 768 + 50304 * 768)
    assert bench.gen_bytes_per_step(c, 50304, B=1, t=0) == weights + 2 * 12 * 1 * 1 * 2 * 768
    assert bench.gen_bytes_per_step(c, 50304, B=16, t=99) - weights == 2 * 12 * 16 * 100 * 2 * 768


def test_config_block_names_the_workload():
    c = synth.WORKLOADS["gpt2_124m"]
    blk = bench.config_block(c, "gpt2_124m")
    assert blk["workload"] == "gpt2_124m" and blk["B"] == 32 and blk["T"] == 1024 and blk["Vp"] == 50304
    assert bench.config_block(c, "gpt2_124m", "rmsnorm")["workload"] == "gpt2_124m_rmsnorm"


def test_palm_flops_per_token_closed_form():
    """6 N + 12 L C T with N = 12 L C^2 + 13 L C + (Vp + maxT) C + 2 C, the GPT-2
    parameter count (per layer: qkv 3C^2 + 3C, attention projection C^2 + C, two
    LayerNorms 4C, fc 4C^2 + 4C, fc projection 4C^2 + C; then wte, wpe and the final
    LayerNorm): 0.860 GFLOP per token for GPT-2 124M at T = 1024."""
    c = synth.WORKLOADS["gpt2_124m"]
    L, C, T, maxT, Vp = c["L"], c["C"], c["T"], c["maxT"], 50304
    n = 12 * L * C * C + 13 * L * C + (Vp + maxT) * C + 2 * C
    assert n == 124_475_904
    assert bench.palm_flops_per_token(c, Vp) == 6 * n + 12 * L * C * T == 860_101_632


def test_cpu_sample_shape_and_extrapolation():
    tiny, big = synth.WORKLOADS["tiny"], synth.WORKLOADS["gpt2_124m"]
    assert bench.sample_shape(tiny, 128) == (tiny["B"], tiny["T"])    # timed in full
    assert bench.sample_shape(big, 128) == (1, 128)
    assert bench.sample_shape(big, 4096) == (1, 1024)
    # a whole-step sample is not scaled: B*T tokens in t_fb + t_adam seconds
    BT = tiny["B"] * tiny["T"]
    assert bench.extrapolated_tokens_per_s(tiny, BT, 2.0, 1.0) == BT / 3.0
    # B*T / 128 samples of fwd+bwd plus one AdamW
    assert bench.extrapolated_tokens_per_s(big, 128, 0.5, 2.0) == 32768 / (256 * 0.5 + 2.0)


def test_oracle_threads_change_no_result():
    """The oracle's OpenMP loops give each thread its own outputs: one thread and several
    give bitwise the same loss and gradients."""
    import numpy as np
    from oracle.oracle import Model, set_threads
    c = synth.WORKLOADS["tiny"]
    L, C, NH, V, maxT = c["L"], c["C"], c["NH"], c["V"], c["maxT"]
    params = synth.init_params(L, C, V, maxT, seed=42)
    inp, tgt = synth.batch(synth.token_stream(c, steps=1), 0, c["B"], c["T"])
    prev = set_threads(0)
    out = []
    try:
        for n in (1, 4):
            assert set_threads(n) == n
            m = Model(L, C, NH, V, maxT)
            m.set_params(params)
            loss = m.forward(inp, tgt)
            m.backward()
            out.append((loss, m.grads()))
    finally:
        set_threads(prev)
    assert out[0][0] == out[1][0]
    assert np.array_equal(out[0][1], out[1][1])


def test_cpu_leg_one_thread_full_tiny_step():
    c = synth.WORKLOADS["tiny"]
    hp = (c["lr"], c["b1"], c["b2"], c["eps"], c["wd"])
    v, used, text = bench.cpu_leg(c, "tiny", "layernorm", 128, hp, variant="f32", threads=1)
    assert v > 0 and used == 1
    assert text.startswith("full step") and "f32 oracle, one thread" in text
