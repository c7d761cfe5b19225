"""Per-operation calls of include/gpt2_ops.h on torch device tensors (marshalling only)."""
from __future__ import annotations

import torch

from . import _native as N


class OpError(RuntimeError):
    pass


def _check(rc):
    if rc != N.GPT2_OK:
        raise OpError(f"{N.STATUS_NAMES.get(rc, rc)}: {N.lib.gpt2_op_last_error().decode()}")


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return N.GPT2_DT_BF16
    if t.dtype == torch.float32:
        return N.GPT2_DT_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _stream():
    return torch.cuda.current_stream().cuda_stream


def bias_grad(dout: torch.Tensor) -> torch.Tensor:
    M, Nn = dout.shape
    out = torch.empty(Nn, dtype=torch.float32, device=dout.device)
    ws_bytes = N.lib.gpt2_op_bias_grad_workspace(M, Nn)
    ws = torch.empty(max(ws_bytes, 4), dtype=torch.uint8, device=dout.device)
    _check(N.lib.gpt2_op_bias_grad(_dt(dout), dout.data_ptr(), M, Nn, out.data_ptr(), ws.data_ptr(),
                                   ws.numel(), _stream()))
    return out


def matmul(A: torch.Tensor, B: torch.Tensor, a_kmajor=True, b_kmajor=True, out_f32=False,
           bias=None, workspace_bytes: int = 64 << 20, tf32: bool = False) -> torch.Tensor:
    """D = A(m,k) B(n,k)^T.  A is (M,K) if a_kmajor else (K,M); B is (N,K) if b_kmajor else (K,N).
    tf32: fp32 operands contracted on the tensor cores as TF32 (fp32 output)."""
    M, K = (A.shape if a_kmajor else A.shape[::-1])
    Nn, K2 = (B.shape if b_kmajor else B.shape[::-1])
    assert K == K2 and A.dtype == B.dtype
    dt = N.GPT2_DT_TF32 if tf32 else _dt(A)
    if tf32:
        assert A.dtype == torch.float32
        out_f32 = True
        workspace_bytes = max(workspace_bytes,
                              N.lib.gpt2_op_matmul_workspace(dt, M, Nn, K, int(a_kmajor), int(b_kmajor)))
    D = torch.empty(M, Nn, dtype=torch.float32 if out_f32 else A.dtype, device=A.device)
    ws = torch.empty(workspace_bytes, dtype=torch.uint8, device=A.device) if workspace_bytes else None
    _check(N.lib.gpt2_op_matmul(dt, M, Nn, K, A.data_ptr(), A.stride(0), int(a_kmajor), B.data_ptr(),
                                B.stride(0), int(b_kmajor), D.data_ptr(), D.stride(0), int(out_f32),
                                None if bias is None else bias.data_ptr(),
                                None if ws is None else ws.data_ptr(), workspace_bytes, _stream()))
    return D


def adamw(p, g, m, v, lr, b1, b2, eps, wd, t, shadow=None):
    _check(N.lib.gpt2_op_adamw(p.data_ptr(), g.data_ptr(), m.data_ptr(), v.data_ptr(),
                               None if shadow is None else shadow.data_ptr(), p.numel(), lr, b1, b2,
                               eps, wd, t, _stream()))


def attention_forward(qkv: torch.Tensor, NH: int):
    B, T, C3 = qkv.shape
    C = C3 // 3
    out = torch.empty(B, T, C, dtype=qkv.dtype, device=qkv.device)
    lse = torch.empty(B, NH, T, dtype=torch.float32, device=qkv.device)
    _check(N.lib.gpt2_op_attention_forward(_dt(qkv), out.data_ptr(), lse.data_ptr(), qkv.data_ptr(),
                                           B, T, C, NH, _stream()))
    return out, lse


def attention_backward(dout, qkv, out, lse, NH: int):
    B, T, C3 = qkv.shape
    C = C3 // 3
    dqkv = torch.empty_like(qkv)
    ws = torch.empty(B * NH * T, dtype=torch.float32, device=qkv.device)
    _check(N.lib.gpt2_op_attention_backward(_dt(qkv), dqkv.data_ptr(), dout.data_ptr(), qkv.data_ptr(),
                                            out.data_ptr(), lse.data_ptr(), B, T, C, NH, ws.data_ptr(),
                                            _stream()))
    return dqkv


def layernorm_forward(x: torch.Tensor, w: torch.Tensor, b: torch.Tensor):
    """x (M,C) -> (out (M,C) like x, mean (M) fp32, rstd (M) fp32)."""
    M, C = x.shape
    out = torch.empty_like(x)
    mean = torch.empty(M, dtype=torch.float32, device=x.device)
    rstd = torch.empty(M, dtype=torch.float32, device=x.device)
    _check(N.lib.gpt2_op_layernorm_forward(_dt(x), out.data_ptr(), mean.data_ptr(), rstd.data_ptr(),
                                           x.data_ptr(), w.data_ptr(), b.data_ptr(), M, C, _stream()))
    return out, mean, rstd


def layernorm_backward(dinp: torch.Tensor, dout, x, w, mean, rstd):
    """dinp (M,C) is accumulated into in place; returns (dw, db) fp32 (C)."""
    M, C = x.shape
    dw = torch.empty(C, dtype=torch.float32, device=x.device)
    db = torch.empty(C, dtype=torch.float32, device=x.device)
    ws_bytes = N.lib.gpt2_op_layernorm_backward_workspace(C)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=x.device)
    _check(N.lib.gpt2_op_layernorm_backward(_dt(x), dinp.data_ptr(), dw.data_ptr(), db.data_ptr(),
                                            dout.data_ptr(), x.data_ptr(), w.data_ptr(), mean.data_ptr(),
                                            rstd.data_ptr(), M, C, ws.data_ptr(), ws_bytes, _stream()))
    return dw, db


def rmsnorm_forward(x: torch.Tensor, w: torch.Tensor):
    """x (M,C) -> (out (M,C) like x, rstd (M) fp32): the microGPT RMSNorm."""
    M, C = x.shape
    out = torch.empty_like(x)
    rstd = torch.empty(M, dtype=torch.float32, device=x.device)
    _check(N.lib.gpt2_op_rmsnorm_forward(_dt(x), out.data_ptr(), rstd.data_ptr(), x.data_ptr(), w.data_ptr(),
                                         M, C, _stream()))
    return out, rstd


def rmsnorm_backward(dinp: torch.Tensor, dout, x, w, rstd):
    """dinp (M,C) is accumulated into in place; returns dw fp32 (C)."""
    M, C = x.shape
    dw = torch.empty(C, dtype=torch.float32, device=x.device)
    ws_bytes = N.lib.gpt2_op_rmsnorm_backward_workspace(C)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=x.device)
    _check(N.lib.gpt2_op_rmsnorm_backward(_dt(x), dinp.data_ptr(), dw.data_ptr(), dout.data_ptr(), x.data_ptr(),
                                          w.data_ptr(), rstd.data_ptr(), M, C, ws.data_ptr(), ws_bytes,
                                          _stream()))
    return dw


def softmax_xent(logits: torch.Tensor, targets: torch.Tensor, V: int, dloss: float, check: bool = True):
    """logits (M,Vp) is overwritten with dlogits; returns the per-row losses (M) fp32."""
    M, Vp = logits.shape
    losses = torch.empty(M, dtype=torch.float32, device=logits.device)
    flags = torch.zeros(1, dtype=torch.int32, device=logits.device) if check else None
    _check(N.lib.gpt2_op_softmax_xent(_dt(logits), logits.data_ptr(), losses.data_ptr(), targets.data_ptr(),
                                      M, V, Vp, dloss, None if flags is None else flags.data_ptr(),
                                      _stream()))
    return losses


def linear_fused(A: torch.Tensor, W: torch.Tensor, epilogue: int, bias=None, R=None, P=None, b_kmajor=True,
                 workspace_bytes: int = 0):
    """bf16 D = A . W^T (W (N,K), b_kmajor) or A . W (W (K,N), not b_kmajor) with a fused epilogue
    (N.GPT2_EPI_*).  Returns D, or (D, gelu(D)) for GPT2_EPI_GELU."""
    M, K = A.shape
    Nn = W.shape[0] if b_kmajor else W.shape[1]
    D = torch.empty(M, Nn, dtype=A.dtype, device=A.device)
    D2 = torch.empty_like(D) if epilogue == N.GPT2_EPI_GELU else None
    ws = torch.empty(workspace_bytes, dtype=torch.uint8, device=A.device) if workspace_bytes else None
    _check(N.lib.gpt2_op_matmul_ex(_dt(A), M, Nn, K, A.data_ptr(), A.stride(0), 1, W.data_ptr(), W.stride(0),
                                   int(b_kmajor), D.data_ptr(), D.stride(0),
                                   None if bias is None else bias.data_ptr(),
                                   None if R is None else R.data_ptr(), 0 if R is None else R.stride(0),
                                   None if D2 is None else D2.data_ptr(), 0 if D2 is None else D2.stride(0),
                                   None if P is None else P.data_ptr(), 0 if P is None else P.stride(0),
                                   epilogue, None if ws is None else ws.data_ptr(), workspace_bytes, _stream()))
    return (D, D2) if D2 is not None else D


def linear_gelu_bwd_bias_grad(A: torch.Tensor, W: torch.Tensor, P: torch.Tensor, b_kmajor=False):
    """bf16 D = (A . W) * gelu'(P) (W (K,N), or W (N,K) with b_kmajor) and dbias = the
    column sums of the stored D (fp32).  Returns (D, dbias)."""
    M, K = A.shape
    Nn = W.shape[0] if b_kmajor else W.shape[1]
    D = torch.empty(M, Nn, dtype=A.dtype, device=A.device)
    dbias = torch.empty(Nn, dtype=torch.float32, device=A.device)
    wsb = N.lib.gpt2_op_matmul_gelu_bwd_bias_grad_workspace(M, Nn)
    ws = torch.empty(max(wsb, 8), dtype=torch.uint8, device=A.device)
    _check(N.lib.gpt2_op_matmul_gelu_bwd_bias_grad(M, Nn, K, A.data_ptr(), A.stride(0), 1, W.data_ptr(),
                                                   W.stride(0), int(b_kmajor), D.data_ptr(), D.stride(0),
                                                   P.data_ptr(), P.stride(0), dbias.data_ptr(), ws.data_ptr(),
                                                   ws.numel(), _stream()))
    return D, dbias


def encoder_forward(tokens: torch.Tensor, wte: torch.Tensor, wpe: torch.Tensor, flags=None):
    """tokens (B,T) int32, wte (V,C), wpe (>=T,C) -> out (B,T,C) like wte."""
    B, T = tokens.shape
    V, C = wte.shape
    out = torch.empty(B, T, C, dtype=wte.dtype, device=wte.device)
    if flags is None:
        flags = torch.zeros(1, dtype=torch.int32, device=wte.device)
    _check(N.lib.gpt2_op_encoder_forward(_dt(wte), out.data_ptr(), tokens.data_ptr(), wte.data_ptr(),
                                         wpe.data_ptr(), B, T, C, V, flags.data_ptr(), _stream()))
    return out


def encoder_backward(dwte: torch.Tensor, dout: torch.Tensor, tokens: torch.Tensor, maxT: int):
    """dwte (V,C) fp32 is accumulated into in place; returns dwpe (maxT,C) fp32."""
    B, T, C = dout.shape
    V = dwte.shape[0]
    dwpe = torch.empty(maxT, C, dtype=torch.float32, device=dout.device)
    ws_bytes = N.lib.gpt2_op_encoder_backward_workspace(B * T, V, C)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dout.device)
    _check(N.lib.gpt2_op_encoder_backward(_dt(dout), dwte.data_ptr(), dwpe.data_ptr(), dout.data_ptr(),
                                          tokens.data_ptr(), B, T, C, V, maxT, ws.data_ptr(), ws.numel(),
                                          _stream()))
    return dwpe


class gemm_tile_rows:
    """Context manager: force the tensor-core GEMM's tiles inside: 128 or 256 rows on one
    SM, or 2 for 256-row tiles computed by a cluster of two CTAs on two SMs."""

    def __init__(self, rows: int):
        self.rows = rows

    def __enter__(self):
        self.prev = N.lib.gpt2_op_gemm_force_tile_rows(self.rows)
        return self

    def __exit__(self, *exc):
        N.lib.gpt2_op_gemm_force_tile_rows(self.prev)


def gemm_last_variant() -> str:
    return N.lib.gpt2_op_gemm_last_variant().decode()
