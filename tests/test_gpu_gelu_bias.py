"""GPU parity of the FC layer's pre-activation gradient with its bias gradient summed in
the same product's epilogue (llm.c annotated listing §1.6 matmul_backward, whose bias
gradient is the sum of the output gradient over positions; §1.10 gelu_backward):
D = (A.W) * gelu'(P) against the oracle's GELU backward of the fp64 product, and dbias
against the fp64 column sums of the D the kernel stored.

Shapes are ragged against the 128/256-row and 256-column tiles and the 32-row groups the
epilogue sums: M = 257 leaves one valid row in the last group, M = 296 leaves the second
CTA of the last pair tile without rows, N = 520 leaves half of the last column tile empty.
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


SHAPES = [(257, 3072, 768), (296, 520, 448), (1000, 768, 96), (2048, 3072, 768), (600, 120, 192)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("tiles", [0, 128, PAIR])
def test_gelu_bwd_bias_grad_fused(torch_cuda, M, N, K, tiles):
    torch = torch_cuda
    from gpt_train_step_arena_b300 import ops
    rng = np.random.default_rng(M * 3 + N * 7 + K + tiles)
    bf = torch.bfloat16
    A = _to(torch, rng.normal(size=(M, K)).astype(np.float32), bf)
    W = _to(torch, (rng.normal(size=(K, N)) / np.sqrt(K)).astype(np.float32), bf)   # (K, N): N-major
    P = _to(torch, (rng.normal(size=(M, N)) * 2).astype(np.float32), bf)
    with ops.gemm_tile_rows(tiles):
        D, db = ops.linear_gelu_bwd_bias_grad(A, W, P)
        variant = ops.gemm_last_variant()
        D2, db2 = ops.linear_gelu_bwd_bias_grad(A, W, P)
    assert "epi=gelu_bwd" in variant and "colsum" in variant, variant
    if tiles == PAIR and N > 128:   # pair tiles are 256 columns wide
        assert variant.startswith("rows=pair256"), variant
    want_D = o64.gelu_backward(_np(P), _np(A) @ _np(W))
    assert _rel(_np(D), want_D) <= 8e-3, variant
    # dbias sums the stored bf16 D in fp32: 32 rows in order, then the ceil(M/32) group
    # sums in a fixed order, each step within 2^-24 of its exact value, so every column is
    # within (31 + M/128 + 34) * 2^-24 * sum |D| of the exact column sum
    d = _np(D)
    want = d.sum(axis=0)
    bound = (31 + M / 128 + 34) * 2.0 ** -24 * np.abs(d).sum(axis=0) + 1e-30
    err = np.abs(_np(db) - want)
    assert np.all(err <= bound), (float(np.max(err / bound)), variant)
    # the separate column-sum pass over the same D agrees within the same bound
    assert np.all(np.abs(_np(ops.bias_grad(D)) - want) <= bound)
    # fixed order: bitwise repeatable
    assert torch.equal(D, D2) and torch.equal(db, db2)


def test_gelu_bwd_bias_grad_no_rows(torch_cuda):
    """M = 0: nothing to sum, dbias is written as zeros."""
    torch = torch_cuda
    from gpt_train_step_arena_b300 import _native as N_
    dbias = torch.full((256,), 7.0, device="cuda")
    rc = N_.lib.gpt2_op_matmul_gelu_bwd_bias_grad(0, 256, 64, None, 64, 1, None, 256, 0, None, 256, None, 256,
                                                  dbias.data_ptr(), None, 0, None)
    torch.cuda.synchronize()
    assert rc == 0 and not dbias.any()
