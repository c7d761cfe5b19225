"""GPU parity of single operations (include/gpt2_ops.h) against the CPU oracle's layer
functions on the same seeded inputs.  Shapes span several tiles and a ragged tail."""
import numpy as np
import pytest

from oracle.oracle import Ops

pytestmark = pytest.mark.gpu

o64 = Ops("f64")
o32 = Ops("f32")


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


# ---------------------------------------------------------------- bias gradient
@pytest.mark.parametrize("M,N", [(1000, 300), (32768 // 16, 3072), (1, 8), (0, 64), (257, 27)])
def test_bias_grad(torch_cuda, M, N):
    torch = torch_cuda
    from gpt_train_step_arena_b300 import ops
    rng = np.random.default_rng(M * 7 + N)
    x = rng.normal(size=(M, N)).astype(np.float32)
    want = x.astype(np.float64).sum(0) if M else np.zeros(N)
    got = _np(ops.bias_grad(_to(torch, x, torch.float32)))
    assert np.allclose(got, want, rtol=1e-5, atol=1e-4 * max(1.0, np.sqrt(M)))
    xb = _to(torch, x, torch.bfloat16)
    want_b = _np(xb).sum(0) if M else np.zeros(N)
    got_b = _np(ops.bias_grad(xb))
    assert np.allclose(got_b, want_b, rtol=1e-5, atol=1e-4 * max(1.0, np.sqrt(M)))
    assert np.array_equal(got_b, _np(ops.bias_grad(xb)))  # fixed summation order


@pytest.mark.parametrize("dt", ["fp32", "bf16"])
def test_bias_grad_unaligned_view(torch_cuda, dt):
    """N % 8 == 0 but dout starts one element off a 16-byte boundary (a column-offset
    view): the kernel must not issue 16-byte loads there, and the sums stay bitwise the
    same as on an aligned copy (same rows in the same order)."""
    torch = torch_cuda
    from gpt_train_step_arena_b300 import ops
    M, N = 777, 512
    tdt = torch.float32 if dt == "fp32" else torch.bfloat16
    rng = np.random.default_rng(77)
    flat = _to(torch, rng.normal(size=M * N + 8).astype(np.float32), tdt)
    view = flat[1:1 + M * N].view(M, N)
    assert view.data_ptr() % 16 != 0
    got = ops.bias_grad(view)
    aligned = ops.bias_grad(view.clone())
    assert torch.equal(got, aligned)
    assert np.allclose(_np(got), _np(view).sum(0), rtol=1e-5, atol=1e-4 * np.sqrt(M))


# ---------------------------------------------------------------- matmul
SHAPES = [(300, 200, 104), (256, 256, 128), (128, 768, 768), (1, 8, 16), (129, 136, 72), (512, 2304, 768)]


def _ref_mm(A, B):
    return A.astype(np.float64) @ B.astype(np.float64).T


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("layout", ["fwd", "dgrad", "wgrad"])
@pytest.mark.parametrize("dt", ["fp32", "bf16"])
def test_matmul_layouts(torch_cuda, M, N, K, layout, dt):
    torch = torch_cuda
    from gpt_train_step_arena_b300 import ops
    rng = np.random.default_rng(M + 3 * N + 7 * K)
    A = rng.normal(size=(M, K)).astype(np.float32)
    B = rng.normal(size=(N, K)).astype(np.float32)
    tdt = torch.float32 if dt == "fp32" else torch.bfloat16
    Ad, Bd = _to(torch, A, tdt), _to(torch, B, tdt)
    A_eff, B_eff = _np(Ad), _np(Bd)  # the values the kernel sees
    if layout == "fwd":        # X . W^T: both K-major
        D = ops.matmul(Ad, Bd, True, True)
    elif layout == "dgrad":    # dY . W: A K-major, B stored (K, N)
        D = ops.matmul(Ad, Bd.t().contiguous(), True, False)
    else:                      # dY^T . X: A stored (K, M), B stored (K, N), fp32 out
        D = ops.matmul(Ad.t().contiguous(), Bd.t().contiguous(), False, False, out_f32=True)
    want = _ref_mm(A_eff, B_eff)
    got = _np(D)
    # fp32 accumulation over K terms; bf16 output adds one rounding (2^-9 relative)
    out_bf16 = dt == "bf16" and layout != "wgrad"
    tol = 8e-3 if out_bf16 else 1e-5
    assert _rel(got, want) <= tol, _rel(got, want)


def test_matmul_bias(torch_cuda):
    torch = torch_cuda
    from gpt_train_step_arena_b300 import ops
    rng = np.random.default_rng(1)
    A = rng.normal(size=(200, 64)).astype(np.float32)
    B = rng.normal(size=(96, 64)).astype(np.float32)
    b = rng.normal(size=96).astype(np.float32)
    D = ops.matmul(_to(torch, A, torch.float32), _to(torch, B, torch.float32), bias=_to(torch, b, torch.float32))
    assert _rel(_np(D), _ref_mm(A, B) + b) <= 1e-5


# ---------------------------------------------------------------- AdamW
def test_adamw_matches_float_oracle_to_ulp(torch_cuda):
    torch = torch_cuda
    from gpt_train_step_arena_b300 import ops
    n = 1_000_003  # not a multiple of 4: exercises the scalar tail
    rng = np.random.default_rng(2)
    p = rng.normal(size=n).astype(np.float32)
    g = (rng.normal(size=n) * 1e-2).astype(np.float32)
    m = (rng.normal(size=n) * 1e-3).astype(np.float32)
    v = np.abs(rng.normal(size=n) * 1e-5).astype(np.float32)
    hp = (6e-4, 0.9, 0.999, 1e-8, 0.1, 7)
    pd, gd, md, vd = (_to(torch, a, torch.float32) for a in (p, g, m, v))
    sh = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    ops.adamw(pd, gd, md, vd, *hp, shadow=sh)
    rp, rm, rv = o32.adamw(p, g, m, v, *hp)
    got = pd.cpu().numpy()
    # p' = p - lr*u: each side rounds p' once (half an ulp of p') and u's few operations
    # (a few ulps of lr*|u| = |p - p'|); fused multiply-adds may differ between the sides.
    step = np.abs(p.astype(np.float64) - rp)
    assert np.all(np.abs(got - rp) <= 2.0 ** -22 * (np.abs(rp) + 4 * step) + 1e-30)
    # m = b1*m + (1-b1)*g can cancel: its rounding error scales with the two terms
    terms = 0.9 * np.abs(m.astype(np.float64)) + 0.1 * np.abs(g.astype(np.float64))
    assert np.all(np.abs(md.cpu().numpy() - rm) <= 2.0 ** -22 * terms + 1e-30)
    assert np.all(np.abs(vd.cpu().numpy() - rv) <= 2.0 ** -22 * np.abs(rv) + 1e-24)
    assert torch.equal(sh, pd.to(torch.bfloat16))


# ---------------------------------------------------------------- attention
@pytest.mark.parametrize("B,T,C,NH", [(2, 77, 64, 4), (1, 1, 32, 2), (2, 130, 128, 2), (1, 256, 768, 12),
                                        (1, 1, 64, 1), (2, 64, 128, 2), (1, 200, 192, 3), (2, 1024, 64, 1)])
@pytest.mark.parametrize("dt", ["fp32", "bf16"])
def test_attention_fwd_bwd(torch_cuda, B, T, C, NH, dt):
    torch = torch_cuda
    from gpt_train_step_arena_b300 import ops
    rng = np.random.default_rng(B * 1000 + T)
    qkv = rng.normal(size=(B, T, 3 * C)).astype(np.float32)
    dy = rng.normal(size=(B, T, C)).astype(np.float32)
    tdt = torch.float32 if dt == "fp32" else torch.bfloat16
    qd, dyd = _to(torch, qkv, tdt), _to(torch, dy, tdt)
    out, lse = ops.attention_forward(qd, NH)
    dq = ops.attention_backward(dyd, qd, out, lse, NH)
    q_eff, dy_eff = _np(qd), _np(dyd)
    ref_out, _, ref_att = o64.attention(q_eff, NH)
    ref_dq = o64.attention_backward(dy_eff, q_eff, ref_att, NH)
    tol_o, tol_g = (1e-5, 1e-4) if dt == "fp32" else (1e-2, 3e-2)
    assert _rel(_np(out), ref_out) <= tol_o
    assert _rel(_np(dq), ref_dq) <= tol_g
    # lse: log of the softmax normaliser of the scaled scores
    hs = C // NH
    q = q_eff[..., :C].reshape(B, T, NH, hs).transpose(0, 2, 1, 3)
    k = q_eff[..., C:2 * C].reshape(B, T, NH, hs).transpose(0, 2, 1, 3)
    s = q @ k.transpose(0, 1, 3, 2) / np.sqrt(hs) + (1 - np.tri(T)) * -1e30
    mx = s.max(-1, keepdims=True)
    ref_lse = (mx + np.log(np.exp(s - mx).sum(-1, keepdims=True)))[..., 0]
    assert np.max(np.abs(_np(lse) - ref_lse)) <= (1e-4 if dt == "fp32" else 2e-2)


# ---------------------------------------------------------------- layernorm
@pytest.mark.parametrize("M,C", [(1000, 768), (37, 768), (300, 100), (1, 256), (513, 1024), (0, 768),
                                 (20000, 768), (5003, 1024)])
@pytest.mark.parametrize("dt", ["fp32", "bf16"])
def test_layernorm_fwd_bwd(torch_cuda, M, C, dt):
    torch = torch_cuda
    from gpt_train_step_arena_b300 import ops
    rng = np.random.default_rng(M * 11 + C)
    x = (rng.normal(size=(M, C)) * 2 + 0.5).astype(np.float32)
    w = (1 + 0.1 * rng.normal(size=C)).astype(np.float32)
    b = (0.1 * rng.normal(size=C)).astype(np.float32)
    dy = rng.normal(size=(M, C)).astype(np.float32)
    acc = rng.normal(size=(M, C)).astype(np.float32)
    tdt = torch.float32 if dt == "fp32" else torch.bfloat16
    xd, dyd, accd = _to(torch, x, tdt), _to(torch, dy, tdt), _to(torch, acc, tdt)
    wd, bd = _to(torch, w, torch.float32), _to(torch, b, torch.float32)
    out, mean, rstd = ops.layernorm_forward(xd, wd, bd)
    acc_before = _np(accd)
    dw, db = ops.layernorm_backward(accd, dyd, xd, wd, mean, rstd)
    torch.cuda.synchronize()
    if M == 0:
        assert np.all(_np(dw) == 0) and np.all(_np(db) == 0)
        return
    x_eff, dy_eff = _np(xd), _np(dyd)
    r_out, r_mean, r_rstd = o64.layernorm(x_eff, w, b)
    r_dx, r_dw, r_db = o64.layernorm_backward(dy_eff, x_eff, w, r_mean, r_rstd)
    assert np.max(np.abs(_np(mean) - r_mean)) <= 1e-5 * (1 + np.max(np.abs(r_mean)))
    assert np.max(np.abs(_np(rstd) / r_rstd - 1)) <= 1e-5
    # fp32: a few roundings per element; bf16: one output rounding (2^-9 relative)
    tol = 1e-5 if dt == "fp32" else 4e-3
    assert _rel(_np(out), r_out) <= tol
    assert _rel(_np(accd) - acc_before, r_dx) <= (1e-5 if dt == "fp32" else 8e-3)
    assert _rel(_np(dw), r_dw) <= 1e-5 and _rel(_np(db), r_db) <= 1e-5
    dw2, db2 = ops.layernorm_backward(_to(torch, acc, tdt), dyd, xd, wd, mean, rstd)
    assert torch.equal(dw, dw2) and torch.equal(db, db2)  # fixed summation order


# ---------------------------------------------------------------- RMSNorm (microGPT variant)
@pytest.mark.parametrize("M,C", [(1000, 768), (37, 768), (300, 100), (1, 256), (513, 1024), (0, 768),
                                 (20000, 768), (5003, 512)])
@pytest.mark.parametrize("dt", ["fp32", "bf16"])
def test_rmsnorm_fwd_bwd(torch_cuda, M, C, dt):
    torch = torch_cuda
    from gpt_train_step_arena_b300 import ops
    rng = np.random.default_rng(M * 13 + C)
    x = (rng.normal(size=(M, C)) * 2 + 0.5).astype(np.float32)   # non-zero mean: not a LayerNorm
    w = (1 + 0.1 * rng.normal(size=C)).astype(np.float32)
    dy = rng.normal(size=(M, C)).astype(np.float32)
    acc = rng.normal(size=(M, C)).astype(np.float32)
    tdt = torch.float32 if dt == "fp32" else torch.bfloat16
    xd, dyd, accd = _to(torch, x, tdt), _to(torch, dy, tdt), _to(torch, acc, tdt)
    wd = _to(torch, w, torch.float32)
    out, rstd = ops.rmsnorm_forward(xd, wd)
    acc_before = _np(accd)
    dw = ops.rmsnorm_backward(accd, dyd, xd, wd, rstd)
    torch.cuda.synchronize()
    if M == 0:
        assert np.all(_np(dw) == 0)
        return
    x_eff, dy_eff = _np(xd), _np(dyd)
    r_out, r_rstd = o64.rmsnorm(x_eff, w)
    r_dx, r_dw = o64.rmsnorm_backward(dy_eff, x_eff, w, r_rstd)
    assert np.max(np.abs(_np(rstd) / r_rstd - 1)) <= 1e-5
    tol = 1e-5 if dt == "fp32" else 4e-3
    assert _rel(_np(out), r_out) <= tol
    assert _rel(_np(accd) - acc_before, r_dx) <= (1e-5 if dt == "fp32" else 8e-3)
    assert _rel(_np(dw), r_dw) <= 1e-5
    dw2 = ops.rmsnorm_backward(_to(torch, acc, tdt), dyd, xd, wd, rstd)
    assert torch.equal(dw, dw2)  # fixed summation order


# ---------------------------------------------------------------- softmax + cross-entropy
@pytest.mark.parametrize("M,V,Vp", [(64, 50257, 50304), (300, 27, 32), (129, 1000, 1000), (5, 1, 8),
                                    (40, 4101, 4104), (3, 9000, 9001)])
@pytest.mark.parametrize("dt", ["fp32", "bf16"])
def test_softmax_xent(torch_cuda, M, V, Vp, dt):
    torch = torch_cuda
    from gpt_train_step_arena_b300 import ops
    rng = np.random.default_rng(M + V)
    logits = (rng.normal(size=(M, Vp)) * 3).astype(np.float32)
    logits[:, V:] = 1e4   # padding columns must be ignored whatever they hold
    tg = rng.integers(0, V, size=M).astype(np.int32)
    tdt = torch.float32 if dt == "fp32" else torch.bfloat16
    ld = _to(torch, logits, tdt)
    l_eff = _np(ld)[:, :V]
    dloss = 1.0 / M
    losses = ops.softmax_xent(ld, torch.from_numpy(tg).to("cuda"), V, dloss)
    _, r_losses, r_dl = o64.cross_entropy(l_eff, tg)
    got_l = _np(losses)
    assert np.max(np.abs(got_l - r_losses)) <= (2e-5 if dt == "fp32" else 1e-4) * max(1.0, np.max(r_losses))
    got_d = _np(ld)
    assert np.all(got_d[:, V:] == 0)
    # relative to the gradient's natural scale (dloss per row): with V = 1 the exact
    # gradient is 0 and the kernel leaves a rounding residue of order 2^-22 * dloss
    scale = max(np.linalg.norm(r_dl), dloss * np.sqrt(M))
    assert np.linalg.norm(got_d[:, :V] - r_dl) <= (1e-5 if dt == "fp32" else 8e-3) * scale


def test_softmax_xent_bad_target(torch_cuda):
    torch = torch_cuda
    from gpt_train_step_arena_b300 import ops
    logits = torch.zeros(4, 64, dtype=torch.bfloat16, device="cuda")
    tg = torch.tensor([0, 1, 64, 3], dtype=torch.int32, device="cuda")
    with pytest.raises(ops.OpError, match="TOKEN"):
        ops.softmax_xent(logits, tg, 64, 0.25)


# ---------------------------------------------------------------- fused linear-layer epilogues
@pytest.mark.parametrize("M,N,K", [(300, 256, 128), (1024, 3072, 768), (257, 768, 3072)])
def test_matmul_fused_epilogues(torch_cuda, M, N, K):
    """The residual, bias+GELU and GELU-backward epilogues of the tensor-core GEMM against the
    oracle's gelu_forward / gelu_backward (llm.c §1.9, §1.10) on the same bf16 operands."""
    torch = torch_cuda
    from gpt_train_step_arena_b300 import ops, _native as N_
    rng = np.random.default_rng(M + N + K)
    bf = torch.bfloat16
    A = _to(torch, rng.normal(size=(M, K)).astype(np.float32) * 0.5, bf)
    W = _to(torch, rng.normal(size=(N, K)).astype(np.float32) / np.sqrt(K), bf)
    bias = _to(torch, rng.normal(size=N).astype(np.float32) * 0.1, torch.float32)
    R = _to(torch, rng.normal(size=(M, N)).astype(np.float32), bf)
    P = _to(torch, rng.normal(size=(M, N)).astype(np.float32) * 2, bf)
    a, w, b, r, pp = _np(A), _np(W), _np(bias), _np(R), _np(P)
    acc = a @ w.T
    # bias + residual
    D = ops.linear_fused(A, W, N_.GPT2_EPI_STORE, bias=bias, R=R)
    assert _rel(_np(D), acc + b + r) <= 8e-3
    # bias + GELU: the pre-activation and its GELU, both rounded once to bf16
    D, G = ops.linear_fused(A, W, N_.GPT2_EPI_GELU, bias=bias)
    pre = acc + b
    assert _rel(_np(D), pre) <= 8e-3
    assert _rel(_np(G), o64.gelu(pre)) <= 8e-3
    # GELU backward in the input-gradient layout (W stored (K, N)): (A . W) * gelu'(P)
    Wt = W.t().contiguous()
    D = ops.linear_fused(A, Wt, N_.GPT2_EPI_GELU_BWD, P=P, b_kmajor=False)
    assert _rel(_np(D), o64.gelu_backward(pp, acc)) <= 8e-3
