"""The TF32 precision mode: fp32 tensors, matrix products on the tensor cores with the
operands read as TF32 (llm.c annotated listing §1.5 matmul_forward / §1.6
matmul_backward contracted with a 10-bit operand mantissa and fp32 accumulation).

Per product: against the fp64 contraction of the same fp32 operands; TF32 keeps 10
mantissa bits, so each operand carries a relative error up to 2^-10 and a K-term sum of
random-sign products a relative-L2 error of about 2^-10; 3e-3 bounds it with margin.
The launched variant must name the TF32 tensor-core kernel (a silent exact-fp32 SIMT
fallback would pass any tolerance).  Whole step: the bf16-mode tolerances (loss 1e-2,
gradients 3e-2 relative-L2 per tensor) against the f64 oracle."""
import numpy as np
import pytest

from .gpu_util import TOL, assert_grads_close, rel_l2

pytestmark = pytest.mark.gpu


def _rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


@pytest.mark.parametrize("M,N,K", [(300, 200, 104), (256, 256, 128), (129, 136, 72), (512, 2304, 768),
                                   (1000, 120, 2112), (64, 50304, 768)])
@pytest.mark.parametrize("layout", ["fwd", "dgrad", "wgrad"])
def test_matmul_tf32_layouts(M, N, K, layout):
    import torch
    from gpt_train_step_arena_b300 import ops
    rng = np.random.default_rng(M + 5 * N + 11 * K)
    A = rng.normal(size=(M, K)).astype(np.float32)
    B = rng.normal(size=(N, K)).astype(np.float32)
    Ad, Bd = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    if layout == "fwd":
        D = ops.matmul(Ad, Bd, True, True, tf32=True)
    elif layout == "dgrad":
        D = ops.matmul(Ad, Bd.t().contiguous(), True, False, tf32=True)
    else:
        D = ops.matmul(Ad.t().contiguous(), Bd.t().contiguous(), False, False, tf32=True)
    variant = ops.gemm_last_variant()
    assert "tf32" in variant, variant
    want = A.astype(np.float64) @ B.astype(np.float64).T
    err = _rel(D.double().cpu().numpy(), want)
    assert err <= 3e-3, (err, variant)
    assert err > 1e-6, "TF32 rounding should be visible; an exact fp32 result means another kernel ran"


def test_matmul_tf32_bias_and_force_256_rows():
    import torch
    from gpt_train_step_arena_b300 import ops
    rng = np.random.default_rng(5)
    A = rng.normal(size=(600, 192)).astype(np.float32)
    W = rng.normal(size=(520, 192)).astype(np.float32)
    b = rng.normal(size=520).astype(np.float32)
    with ops.gemm_tile_rows(256):
        D = ops.matmul(torch.from_numpy(A).cuda(), torch.from_numpy(W).cuda(), bias=torch.from_numpy(b).cuda(),
                       tf32=True)
        variant = ops.gemm_last_variant()
    assert variant.startswith("rows=256") and "tf32" in variant, variant
    want = A.astype(np.float64) @ W.astype(np.float64).T + b
    assert _rel(D.double().cpu().numpy(), want) <= 3e-3


def test_fp32_dtype_stays_exact():
    """GPT2_DT_F32 (the strict fp32 mode) must not take the TF32 path."""
    import torch
    from gpt_train_step_arena_b300 import ops
    rng = np.random.default_rng(6)
    A = rng.normal(size=(300, 256)).astype(np.float32)
    B = rng.normal(size=(200, 256)).astype(np.float32)
    D = ops.matmul(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda())
    assert ops.gemm_last_variant() == "simt"
    assert _rel(D.double().cpu().numpy(), A.astype(np.float64) @ B.astype(np.float64).T) <= 1e-6


@pytest.mark.parametrize("name", ["tiny", "gpt2_124m_small"])
def test_tf32_one_step(name):
    from .test_gpu_parity import _run_one_step
    from gpt_train_step_arena_b300.model import GPT2
    r = _run_one_step(GPT2, name, "tf32")
    tol = TOL["bf16"]
    L, C, V, maxT = r["shape"]
    assert np.array_equal(r["tok_back"], r["inp"]) and np.array_equal(r["tgt_back"], r["tgt"])
    assert abs(r["loss"] - r["ref_loss"]) <= tol["loss"] * abs(r["ref_loss"]), (r["loss"], r["ref_loss"])
    assert rel_l2(r["logits"], r["ref_logits"]) <= 3e-2
    assert_grads_close(r["grads"], r["ref_grads"], L, C, V, maxT, tol["grads"])
