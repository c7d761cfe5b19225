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


def test_bias_grad_noalloc_matches_workspace_entry_point():
    import torch
    from gpt_train_step_arena_b300 import _native as N

    stream = torch.cuda.current_stream().cuda_stream
    rng = np.random.default_rng(2024)
    # two calls in a row, of different shape and dtype
    for M, Nn, dt in ((4096, 3072, torch.bfloat16), (1000, 300, torch.float32)):
        x = torch.from_numpy(rng.normal(size=(M, Nn)).astype(np.float32)).to("cuda").to(dt)
        code = N.GPT2_DT_BF16 if dt == torch.bfloat16 else N.GPT2_DT_F32
        ws_bytes = N.lib.gpt2_op_bias_grad_workspace(M, Nn)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        want = torch.empty(Nn, dtype=torch.float32, device="cuda")
        got = torch.full((Nn,), float("nan"), dtype=torch.float32, device="cuda")
        assert N.lib.gpt2_op_bias_grad(code, x.data_ptr(), M, Nn, want.data_ptr(), ws.data_ptr(),
                                       ws_bytes, stream) == N.GPT2_OK
        rc = N.lib.gpt2_op_bias_grad_noalloc(code, x.data_ptr(), M, Nn, got.data_ptr(), stream)
        assert rc == N.GPT2_OK, N.lib.gpt2_op_last_error().decode()
        torch.cuda.synchronize()
        w, g = want.cpu().numpy(), got.cpu().numpy()
        assert np.allclose(g, w, rtol=1e-5, atol=1e-4 * np.sqrt(M))
        assert np.array_equal(g, w)  # same kernels, same summation order


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
