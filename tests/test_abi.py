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
