"""GPU parity of the tensor-core GEMM run by clusters of two CTAs on two SMs (256-row
tiles, 128 rows and half of every B tile per SM, cta_group::2 MMAs issued by the leader),
against the fp64 contraction of the bf16 operands the kernel sees (llm.c annotated listing
§1.5 matmul_forward, §1.6 matmul_backward) and the oracle's GELU (§1.9, §1.10).

Shapes are ragged against the pair tile (M and N multiples of 8, as the M-major and N-major
layouts need): M = 296 leaves the second CTA of the last pair
with no valid row at all, N = 520 leaves the second CTA's half of the last B tile empty,
K = 2112 splits the fp32 weight gradient.
"""
import numpy as np
import pytest

from oracle.oracle import Ops

pytestmark = pytest.mark.gpu

o64 = Ops("f64")
PAIR = 2


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    assert torch.cuda.is_available()
    return torch


def _to(torch, a, dtype):
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda").to(dtype)


def _np(t):
    return t.float().cpu().numpy().astype(np.float64)


def _rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


SHAPES = [(296, 520, 448), (600, 520, 2112), (1000, 768, 96), (264, 1000, 192), (2048, 2304, 768)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("layout", ["fwd", "dgrad", "wgrad"])
def test_matmul_pair_tiles(torch_cuda, M, N, K, layout):
    torch = torch_cuda
    from gpt_train_step_arena_b300 import ops
    rng = np.random.default_rng(M * 7 + N * 5 + K)
    A = rng.normal(size=(M, K)).astype(np.float32)
    B = rng.normal(size=(N, K)).astype(np.float32)
    Ad, Bd = _to(torch, A, torch.bfloat16), _to(torch, B, torch.bfloat16)
    want = _np(Ad) @ _np(Bd).T
    with ops.gemm_tile_rows(PAIR):
        if layout == "fwd":
            D = ops.matmul(Ad, Bd, True, True)
        elif layout == "dgrad":
            D = ops.matmul(Ad, Bd.t().contiguous(), True, False)
        else:
            D = ops.matmul(Ad.t().contiguous(), Bd.t().contiguous(), False, False, out_f32=True)
        variant = ops.gemm_last_variant()
    assert variant.startswith("rows=pair256"), variant
    # fp32 accumulation; a bf16 output adds one rounding (2^-9 relative)
    tol = 1e-5 if layout == "wgrad" else 8e-3
    assert _rel(_np(D), want) <= tol, (_rel(_np(D), want), variant)
    # every row block of 128 (each CTA's half of every pair tile) and the ragged tails
    got = _np(D)
    for r0 in range(0, got.shape[0], 128):
        blk = slice(r0, min(got.shape[0], r0 + 128))
        assert _rel(got[blk], want[blk]) <= 2 * tol, (r0, variant)


@pytest.mark.parametrize("M,N,K", [(300, 520, 192), (1024, 3072, 768), (257, 768, 3072)])
def test_matmul_pair_fused_epilogues(torch_cuda, M, N, K):
    """Bias + residual, bias + GELU and the GELU-backward epilogue on pair tiles."""
    torch = torch_cuda
    from gpt_train_step_arena_b300 import ops, _native as N_
    rng = np.random.default_rng(M + 3 * N + K)
    bf = torch.bfloat16
    A = _to(torch, rng.normal(size=(M, K)).astype(np.float32) * 0.5, bf)
    W = _to(torch, rng.normal(size=(N, K)).astype(np.float32) / np.sqrt(K), bf)
    bias = _to(torch, rng.normal(size=N).astype(np.float32) * 0.1, torch.float32)
    R = _to(torch, rng.normal(size=(M, N)).astype(np.float32), bf)
    P = _to(torch, rng.normal(size=(M, N)).astype(np.float32) * 2, bf)
    a, w, b, r, pp = _np(A), _np(W), _np(bias), _np(R), _np(P)
    acc = a @ w.T
    with ops.gemm_tile_rows(PAIR):
        D = ops.linear_fused(A, W, N_.GPT2_EPI_STORE, bias=bias, R=R)
        assert ops.gemm_last_variant().startswith("rows=pair256")
        assert _rel(_np(D), acc + b + r) <= 8e-3
        D, G = ops.linear_fused(A, W, N_.GPT2_EPI_GELU, bias=bias)
        assert ops.gemm_last_variant().startswith("rows=pair256")
        pre = acc + b
        assert _rel(_np(D), pre) <= 8e-3
        assert _rel(_np(G), o64.gelu(pre)) <= 8e-3
        Wt = W.t().contiguous()
        D = ops.linear_fused(A, Wt, N_.GPT2_EPI_GELU_BWD, P=P, b_kmajor=False)
        assert ops.gemm_last_variant().startswith("rows=pair256")
        assert _rel(_np(D), o64.gelu_backward(pp, acc)) <= 8e-3


def test_matmul_pair_repeatable(torch_cuda):
    """Two runs of a pair product are bitwise equal (fixed accumulation order)."""
    torch = torch_cuda
    from gpt_train_step_arena_b300 import ops
    rng = np.random.default_rng(5)
    A = _to(torch, rng.normal(size=(1500, 768)).astype(np.float32), torch.bfloat16)
    B = _to(torch, rng.normal(size=(2304, 768)).astype(np.float32), torch.bfloat16)
    with ops.gemm_tile_rows(PAIR):
        D1 = ops.matmul(A, B, True, True)
        D2 = ops.matmul(A, B, True, True)
    assert torch.equal(D1, D2)


def test_pair_whole_step_matches_default_tiles(torch_cuda):
    """A whole bf16 training step (GPT-2 small shapes, B=2, T=256) with every product on
    pair tiles agrees with the per-shape default within bf16 rounding."""
    torch = torch_cuda
    from gpt_train_step_arena_b300 import ops, synth
    from gpt_train_step_arena_b300.model import GPT2
    L, C, NH, V, maxT = 2, 768, 12, 50257, 1024
    params = synth.init_params(L, C, V, maxT, seed=7)
    rng = np.random.default_rng(8)
    inp = rng.integers(0, V, size=(2, 256)).astype(np.int32)
    tgt = rng.integers(0, V, size=(2, 256)).astype(np.int32)
    out = {}
    for mode in (0, PAIR):
        with ops.gemm_tile_rows(mode):
            g = GPT2(L, C, NH, V, maxT, precision="bf16")
            g.set_params(params)
            loss = g.forward(inp, tgt)
            g.backward()
            out[mode] = (loss, g.grads())
            g.close()
    (l0, g0), (l1, g1) = out[0], out[PAIR]
    assert abs(l0 - l1) <= 1e-3 * abs(l0)
    assert _rel(np.asarray(g1, dtype=np.float64), np.asarray(g0, dtype=np.float64)) <= 2e-2
