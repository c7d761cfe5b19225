"""GPU parity of the kernel variants that only the full-size training step selects,
against the CPU oracle (or, for products, the exact fp64 contraction of the operands the
kernel sees):

* the tensor-core GEMM with 256-row tiles on one SM (two 128-row accumulator halves
  sharing each B stage), which the per-shape choice takes for the LM-head gradients and
  the long-K input gradients at B=32, T=1024: forced on small ragged shapes in every
  operand layout; and the 256-row tiles on CTA pairs that it takes for the forward
  products, reached naturally on an LM-head-sized forward product;
* the encoder backward's long buckets (positions of one id split into segments summed in
  a second pass) and its multi-chunk ranking, at M = 32,768 Zipf(1.1) ids over the GPT-2
  vocabulary, where id 0 alone holds thousands of positions;
* whole-step batch slices at the benchmark's sequence length: GPT-2 124M at B=2,
  T=1024 and GPT-2 350M at B=1, T=1024, bf16 mixed precision, against the f64 oracle.
"""
import numpy as np
import pytest

from gpt_train_step_arena_b300 import synth
from oracle.oracle import Model as Oracle
from oracle.oracle import Ops

from .gpu_util import TOL, assert_grads_close, cfg_shape

pytestmark = pytest.mark.gpu

o64 = Ops("f64")


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


# ---------------------------------------------------------------- 256-row GEMM tiles
# (M, N, K): ragged against the 256-row, 128/256-column and 64-deep tiles (multiples of 8
# only, which the M-major and N-major layouts need); K = 448 keeps the weight gradient
# unsplit (7 K blocks), K = 2112 splits it; N = 120 takes 128-column tiles.
FORCED = [(600, 520, 2112), (304, 136, 448), (264, 1000, 96), (1000, 120, 2112)]


@pytest.mark.parametrize("M,N,K", FORCED)
@pytest.mark.parametrize("layout", ["fwd", "dgrad", "wgrad"])
def test_matmul_256_row_tiles(torch_cuda, M, N, K, layout):
    torch = torch_cuda
    from gpt_train_step_arena_b300 import ops
    rng = np.random.default_rng(M * 5 + N * 3 + K)
    A = rng.normal(size=(M, K)).astype(np.float32)
    B = rng.normal(size=(N, K)).astype(np.float32)
    Ad, Bd = _to(torch, A, torch.bfloat16), _to(torch, B, torch.bfloat16)
    want = _np(Ad) @ _np(Bd).T
    with ops.gemm_tile_rows(256):
        if layout == "fwd":
            D = ops.matmul(Ad, Bd, True, True)
        elif layout == "dgrad":
            D = ops.matmul(Ad, Bd.t().contiguous(), True, False)
        else:
            D = ops.matmul(Ad.t().contiguous(), Bd.t().contiguous(), False, False, out_f32=True)
        variant = ops.gemm_last_variant()
    assert variant.startswith("rows=256"), variant
    if layout == "wgrad" and K == 448:
        assert "splits=1" in variant, variant
    # fp32 accumulation; a bf16 output adds one rounding (2^-9 relative)
    tol = 1e-5 if layout == "wgrad" else 8e-3
    assert _rel(_np(D), want) <= tol, (_rel(_np(D), want), variant)


def test_matmul_256_row_tiles_bias(torch_cuda):
    """The forward product with a bias on 256-row tiles (the QKV and FC shapes' epilogue)."""
    torch = torch_cuda
    from gpt_train_step_arena_b300 import ops
    rng = np.random.default_rng(11)
    A = _to(torch, rng.normal(size=(700, 192)).astype(np.float32), torch.bfloat16)
    W = _to(torch, rng.normal(size=(520, 192)).astype(np.float32), torch.bfloat16)
    b = _to(torch, rng.normal(size=520).astype(np.float32), torch.float32)
    with ops.gemm_tile_rows(256):
        D = ops.matmul(A, W, bias=b)
        variant = ops.gemm_last_variant()
    assert variant.startswith("rows=256"), variant
    assert _rel(_np(D), _np(A) @ _np(W).T + _np(b)) <= 8e-3


def test_matmul_lm_head_size_takes_pair_tiles(torch_cuda):
    """LM-head forward shape (M = 6272 rows, Vp = 50304, C = 768): the per-shape choice
    itself picks 256-row tiles on CTA pairs; rows sampled across every row tile and the
    ragged last one are checked against the fp64 product."""
    torch = torch_cuda
    from gpt_train_step_arena_b300 import ops
    M, N, K = 6272, 50304, 768
    rng = np.random.default_rng(3)
    A = _to(torch, rng.normal(size=(M, K)).astype(np.float32), torch.bfloat16)
    W = _to(torch, (rng.normal(size=(N, K)) * 0.02).astype(np.float32), torch.bfloat16)
    D = ops.matmul(A, W)
    variant = ops.gemm_last_variant()
    assert variant.startswith("rows=pair256"), variant
    rows = np.unique(np.concatenate([np.arange(0, M, 97), [M - 1, M - 2, 255, 256, 511]]))
    got = _np(D[torch.from_numpy(rows).to("cuda")])
    want = _np(A[torch.from_numpy(rows).to("cuda")]) @ _np(W).T
    assert _rel(got, want) <= 8e-3
    # every column block, including the last (50304 = 196.5 x 256)
    for c0 in range(0, N, 256):
        blk = slice(c0, min(N, c0 + 256))
        assert _rel(got[:, blk], want[:, blk]) <= 1e-2, c0


# ---------------------------------------------------------------- encoder
@pytest.mark.parametrize("dt", ["fp32", "bf16"])
def test_encoder_forward(torch_cuda, dt):
    torch = torch_cuda
    from gpt_train_step_arena_b300 import ops
    B, T, C, V, maxT = 3, 77, 96, 1000, 128
    rng = np.random.default_rng(9)
    wte = rng.normal(size=(V, C)).astype(np.float32)
    wpe = rng.normal(size=(maxT, C)).astype(np.float32)
    tok = synth.zipf_stream(V, B * T, seed=10).reshape(B, T)
    tdt = torch.float32 if dt == "fp32" else torch.bfloat16
    wted, wped = _to(torch, wte, tdt), _to(torch, wpe, tdt)
    out = ops.encoder_forward(torch.from_numpy(tok).to("cuda"), wted, wped)
    want = o64.encoder(tok, _np(wted), _np(wped))
    got = _np(out)
    if dt == "fp32":
        assert np.max(np.abs(got - want)) <= 1e-6 * np.max(np.abs(want))
    else:   # one bf16 rounding of the exact sum
        assert np.max(np.abs(got - want) / np.maximum(np.abs(want), 1e-30)) <= 2.0 ** -8


@pytest.mark.parametrize("dt", ["fp32", "bf16"])
def test_encoder_backward_zipf_full_batch(torch_cuda, dt):
    """M = 32,768 Zipf(1.1) ids over V = 50,257 (the 124M step's batch): many chunks of
    the counting sort, and buckets far longer than one segment."""
    torch = torch_cuda
    from gpt_train_step_arena_b300 import ops
    B, T, C, V, maxT = 32, 1024, 768, 50257, 1024
    tok = synth.zipf_stream(V, B * T, seed=1337).reshape(B, T)
    counts = np.bincount(tok.reshape(-1), minlength=V)
    assert counts.max() > 2000 and (counts > 64).sum() > 20   # long buckets are exercised
    rng = np.random.default_rng(12)
    dout = rng.normal(size=(B, T, C)).astype(np.float32)
    tdt = torch.float32 if dt == "fp32" else torch.bfloat16
    doutd = _to(torch, dout, tdt)
    tokd = torch.from_numpy(tok).to("cuda")
    init = (rng.normal(size=(V, C)) * 0.01).astype(np.float32)   # the LM head's share, added onto
    dwte = _to(torch, init, torch.float32)
    dwpe = ops.encoder_backward(dwte, doutd, tokd, maxT)
    ref_wte, ref_wpe = o64.encoder_backward(_np(doutd), tok, V, maxT)
    got_wte = _np(dwte) - init
    # fp32 sums in a fixed order: n terms summed in segments of 64 then segment by segment
    # carry a relative error of about 2^-24 (sqrt(64/2) + sqrt(n/128)), under 1e-6 for the
    # longest bucket here
    assert _rel(got_wte, ref_wte) <= 4e-6
    assert _rel(_np(dwpe), ref_wpe) <= 4e-6
    heavy = np.argsort(counts)[-5:]
    assert _rel(got_wte[heavy], ref_wte[heavy]) <= 4e-6
    assert not got_wte[counts == 0].any()                      # untouched rows keep their values
    dwte2 = _to(torch, init, torch.float32)
    dwpe2 = ops.encoder_backward(dwte2, doutd, tokd, maxT)
    assert torch.equal(dwte, dwte2) and torch.equal(dwpe, dwpe2)   # bitwise reproducible


# ---------------------------------------------------------------- whole-step batch slices
def _slice_step(name, B, T):
    from gpt_train_step_arena_b300.model import GPT2
    c = synth.WORKLOADS[name]
    L, C, NH, V, maxT = cfg_shape(name)
    params = synth.init_params(L, C, V, maxT, seed=42)
    inp, tgt = synth.batch(synth.token_stream(c, steps=1), 0, B, T)   # first B rows of step 1
    g = GPT2(L, C, NH, V, maxT, precision="bf16")
    g.set_params(params)
    loss = g.forward(inp, tgt)
    g.backward()
    grads = g.grads()
    g.close()
    o = Oracle(L, C, NH, V, maxT)
    o.set_params(params)
    ref_loss = o.forward(inp, tgt)
    o.backward()
    ref_grads = o.grads()
    del o
    return loss, ref_loss, grads, ref_grads, (L, C, V, maxT)


@pytest.mark.slow
def test_gpt2_124m_slice_b2_t1024_bf16():
    loss, ref_loss, grads, ref_grads, (L, C, V, maxT) = _slice_step("gpt2_124m", 2, 1024)
    tol = TOL["bf16"]
    assert abs(loss - ref_loss) <= tol["loss"] * ref_loss, (loss, ref_loss)
    assert_grads_close(grads, ref_grads, L, C, V, maxT, tol["grads"])


@pytest.mark.slow
def test_gpt2_350m_slice_b1_t1024_bf16():
    loss, ref_loss, grads, ref_grads, (L, C, V, maxT) = _slice_step("gpt2_350m", 1, 1024)
    tol = TOL["bf16"]
    assert abs(loss - ref_loss) <= tol["loss"] * ref_loss, (loss, ref_loss)
    assert_grads_close(grads, ref_grads, L, C, V, maxT, tol["grads"])
