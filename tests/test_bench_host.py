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
