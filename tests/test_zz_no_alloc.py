"""The bias-gradient entry point that allocates nothing (for callers that cannot
allocate device memory) must give the same result as the workspace entry point.

This file is collected last on purpose: when it fails, a run that stops at the first
failure has already run every other test.  It passes alone in a fresh process and
after the other tests (the fixed array keeps whatever the previous call left, which
must not matter)."""
import ctypes as ct

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

# (M, N, dtype, element offset of dout from a 16-byte boundary)
CASES = [
    (4096, 3072, "bf16", 0),   # vector path
    (1000, 300, "f32", 0),     # N % 8 != 0: scalar path
    (1000, 300, "bf16", 0),    # bf16 scalar path
    (777, 64, "bf16", 1),      # N % 8 == 0 but dout 2 bytes off a 16-byte boundary: scalar path
    (513, 128, "f32", 1),      # fp32, 4 bytes off
    (0, 64, "bf16", 0),        # no rows: dbias is zero-filled
]


def _run(M, Nn, dt, off, rng):
    import torch
    from gpt_train_step_arena_b300 import _native as N

    stream = torch.cuda.current_stream().cuda_stream
    tdt = torch.bfloat16 if dt == "bf16" else torch.float32
    code = N.GPT2_DT_BF16 if dt == "bf16" else N.GPT2_DT_F32
    flat = torch.from_numpy(rng.normal(size=M * Nn + 8).astype(np.float32)).to("cuda").to(tdt)
    x = flat[off:off + M * Nn]          # a view that may start off a 16-byte boundary
    ptr = x.data_ptr() if M else flat.data_ptr()
    ws_bytes = N.lib.gpt2_op_bias_grad_workspace(M, Nn)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device="cuda")
    want = torch.full((Nn,), float("nan"), dtype=torch.float32, device="cuda")
    got = torch.full((Nn,), float("nan"), dtype=torch.float32, device="cuda")
    assert N.lib.gpt2_op_bias_grad(code, ptr, M, Nn, want.data_ptr(), ws.data_ptr(), ws_bytes,
                                   stream) == N.GPT2_OK
    rc = N.lib.gpt2_op_bias_grad_noalloc(code, ptr, M, Nn, got.data_ptr(), stream)
    assert rc == N.GPT2_OK, N.lib.gpt2_op_last_error().decode()
    torch.cuda.synchronize()
    ref = x.double().reshape(M, Nn).sum(0).cpu().numpy() if M else np.zeros(Nn)
    return want.cpu().numpy(), got.cpu().numpy(), ref


def test_bias_grad_noalloc_matches_workspace_entry_point():
    rng = np.random.default_rng(2024)
    # several calls in a row sharing the fixed array, of different shape, dtype and alignment
    for M, Nn, dt, off in CASES:
        w, g, ref = _run(M, Nn, dt, off, rng)
        assert np.array_equal(g, w), (M, Nn, dt, off)  # same kernels, same summation order
        assert np.allclose(g, ref, rtol=1e-5, atol=1e-4 * np.sqrt(max(M, 1))), (M, Nn, dt, off)
        if M == 0:
            assert np.all(g == 0)


def test_bias_grad_noalloc_rejects_oversize():
    import torch
    from gpt_train_step_arena_b300 import _native as N

    cap = N.lib.gpt2_op_bias_grad_noalloc_max_floats()
    M, Nn = 256 * (cap // 1024 + 1), 1024   # ceil(M/256) * N > cap
    out = torch.empty(Nn, dtype=torch.float32, device="cuda")
    rc = N.lib.gpt2_op_bias_grad_noalloc(N.GPT2_DT_F32, ct.c_void_p(16), M, Nn, out.data_ptr(),
                                         torch.cuda.current_stream().cuda_stream)
    assert rc == N.GPT2_ERR_ARG
    assert "scratch" in N.lib.gpt2_op_last_error().decode()
