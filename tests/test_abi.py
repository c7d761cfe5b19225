"""CPU checks of the boundary: the C-ABI library builds, loads, and exports every
entry point that include/*.h declares (no compute call: there is no GPU here)."""
import glob
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b(gpt2\w*)\s*\(", text))
    return names


def test_headers_declare_the_boundary():
    names = _declared()
    for required in ("gpt2_build", "gpt2_forward", "gpt2_backward", "gpt2_update", "gpt2_free"):
        assert required in names


def test_library_exports_every_declared_symbol():
    from gpt_train_step_arena_b300 import build as b
    lib = b.build()
    out = subprocess.run(["nm", "-D", "--defined-only", lib], capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    missing = _declared() - exported
    assert not missing, missing


def test_binding_declares_every_header_symbol():
    from gpt_train_step_arena_b300 import _native
    assert _declared() <= set(_native.SIGNATURES), _declared() - set(_native.SIGNATURES)
    for name in _native.SIGNATURES:
        assert hasattr(_native.lib, name)


def test_product_path_does_not_reference_the_oracle():
    pkg = os.path.join(ROOT, "gpt_train_step_arena_b300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert not re.search(r"^\s*(import|from)\s+oracle|liboracle|gpt2_oracle", text, re.M), f


def test_build_rejects_bad_arguments_before_touching_the_device():
    """Argument checks of gpt2_build_norm run on the host: no CUDA call is made, so this
    needs no GPU."""
    import ctypes as ct
    from gpt_train_step_arena_b300 import _native as N
    st = ct.c_int(0)
    assert not N.lib.gpt2_build_norm(1, 16, 4, 27, 16, N.GPT2_FP32, 7, ct.byref(st))   # unknown norm
    assert st.value == N.GPT2_ERR_ARG and b"norm" in N.lib.gpt2_last_build_error()
    assert not N.lib.gpt2_build_norm(1, 16, 5, 27, 16, N.GPT2_FP32, N.GPT2_RMSNORM, ct.byref(st))  # C % H
    assert st.value == N.GPT2_ERR_ARG
    assert not N.lib.gpt2_build_ex(1, 16, 4, 27, 16, 3, ct.byref(st))                 # unknown precision
    assert st.value == N.GPT2_ERR_ARG


def test_gelu_bwd_bias_grad_rejects_bad_arguments_on_the_host():
    """gpt2_op_matmul_gelu_bwd_bias_grad checks sizes, pointers and the workspace before
    any CUDA call (no GPU needed); N = 0 is an empty call."""
    from gpt_train_step_arena_b300 import _native as N
    f = N.lib.gpt2_op_matmul_gelu_bwd_bias_grad
    M, Nn, K = 300, 520, 448
    need = N.lib.gpt2_op_matmul_gelu_bwd_bias_grad_workspace(M, Nn)
    # the larger of ceil(M/32) x N group sums and the column-sum pass's partials, fp32
    assert need >= ((M + 31) // 32) * Nn * 4
    assert N.lib.gpt2_op_matmul_gelu_bwd_bias_grad_workspace(0, Nn) == 0
    p = 4096   # never dereferenced: every call below stops at an argument check
    args = dict(A=p, lda=K, ak=1, B=p, ldb=Nn, bk=0, D=p, ldd=Nn, P=p, ldp=Nn, db=p, ws=p, wsb=need)

    def call(M=M, Nn=Nn, K=K, **kw):
        a = dict(args, **kw)
        return f(M, Nn, K, a["A"], a["lda"], a["ak"], a["B"], a["ldb"], a["bk"], a["D"], a["ldd"], a["P"],
                 a["ldp"], a["db"], a["ws"], a["wsb"], None)

    assert call(M=-1) == N.GPT2_ERR_ARG
    assert call(Nn=0) == N.GPT2_OK
    assert call(db=None) == N.GPT2_ERR_ARG
    assert call(P=None) == N.GPT2_ERR_ARG
    assert call(ws=None) == N.GPT2_ERR_ARG
    assert call(wsb=need - 4) == N.GPT2_ERR_ARG and b"workspace" in N.lib.gpt2_op_last_error()
    assert call(ws=p + 4) == N.GPT2_ERR_ARG      # not 8-byte aligned
