"""Helpers shared by the GPU parity tests: run the CUDA library and the oracle on the
same seeded inputs and compare with the tolerances of the training-step contract."""
from __future__ import annotations

import numpy as np

from gpt_train_step_arena_b300 import synth

# Tolerances (loss relative, logits relative-L2 and max-abs, gradients relative-L2 per
# parameter tensor) of the two precision modes.
TOL = {
    "fp32": dict(loss=1e-5, logits=1e-4, grads=1e-3),
    "bf16": dict(loss=1e-2, logits=None, grads=3e-2),
}


def cfg_shape(name):
    c = synth.WORKLOADS[name]
    return c["L"], c["C"], c["NH"], c["V"], c["maxT"]


def split(flat, L, C, V, maxT):
    sizes = synth.param_sizes(L, C, V, maxT)
    return dict(zip(synth.PARAM_NAMES, np.split(np.asarray(flat, np.float64), np.cumsum(sizes)[:-1])))


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    nb = np.linalg.norm(b)
    if nb == 0:
        return float(np.linalg.norm(a))
    return float(np.linalg.norm(a - b) / nb)


def per_tensor_errors(got, want, L, C, V, maxT):
    g, w = split(got, L, C, V, maxT), split(want, L, C, V, maxT)
    return {k: rel_l2(g[k], w[k]) for k in synth.PARAM_NAMES}


def assert_grads_close(got, want, L, C, V, maxT, tol):
    errs = per_tensor_errors(got, want, L, C, V, maxT)
    bad = {k: e for k, e in errs.items() if not e <= tol}
    assert not bad, f"gradient tensors over {tol}: {bad}"
    return errs
