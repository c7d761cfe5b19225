"""ctypes wrapper over the CPU oracle (test infrastructure only).

Only tests, the smoke check and the benchmark's CPU-baseline leg import this
module.  The CUDA library never does.
"""
from __future__ import annotations

import ctypes as ct
import os

import numpy as np

from . import build as _build

_LIBS: dict = {}


def _lib(variant: str):
    if variant not in _LIBS:
        _build.build()
        lib = ct.CDLL(_build.lib_path(variant))
        R = ct.c_double if variant == "f64" else ct.c_float
        P = ct.c_void_p
        i, z = ct.c_int, ct.c_size_t
        sigs = {
            "or_encoder_forward": (None, [P, P, P, P, i, i, i]),
            "or_encoder_backward": (None, [P, P, P, P, i, i, i]),
            "or_layernorm_forward": (None, [P, P, P, P, P, P, i, i, i]),
            "or_layernorm_backward": (None, [P, P, P, P, P, P, P, P, i, i, i]),
            "or_rmsnorm_forward": (None, [P, P, P, P, i, i, i]),
            "or_rmsnorm_backward": (None, [P, P, P, P, P, P, i, i, i]),
            "or_matmul_forward": (None, [P, P, P, P, i, i, i, i]),
            "or_matmul_backward": (None, [P, P, P, P, P, P, i, i, i, i]),
            "or_attention_forward": (None, [P, P, P, P, i, i, i, i]),
            "or_attention_backward": (None, [P, P, P, P, P, P, i, i, i, i]),
            "or_gelu_forward": (None, [P, P, z]),
            "or_gelu_backward": (None, [P, P, P, z]),
            "or_residual_forward": (None, [P, P, P, z]),
            "or_residual_backward": (None, [P, P, P, z]),
            "or_softmax_forward": (None, [P, P, i, i, i]),
            "or_crossentropy_forward": (None, [P, P, P, i, i, i]),
            "or_crossentropy_softmax_backward": (None, [P, P, P, P, i, i, i]),
            "or_adamw": (i, [P, P, P, P, z, R, R, R, R, R, i]),
            "or_build": (P, [i, i, i, i, i]),
            "or_build_ex": (P, [i, i, i, i, i, i]),
            "or_num_params": (z, [P]),
            "or_num_acts": (z, [P]),
            "or_param_sizes": (None, [P, P]),
            "or_set_params": (None, [P, P]),
            "or_get_params": (None, [P, P]),
            "or_get_grads": (i, [P, P]),
            "or_get_opt_state": (i, [P, P, P]),
            "or_get_logits": (i, [P, P]),
            "or_get_losses": (i, [P, P]),
            "or_get_dencoded": (i, [P, P]),
            "or_forward": (i, [P, P, P, i, i, P]),
            "or_zero_grad": (None, [P]),
            "or_backward": (i, [P]),
            "or_update": (i, [P, R, R, R, R, R, i]),
            "or_free": (None, [P]),
            "or_real_bytes": (i, []),
            "or_set_threads": (i, [i]),
            "or_release_acts": (None, [P]),
            "or_sample_mult": (i, [P, i, R]),
            "or_generate": (i, [P, P, i, i, i, R, P, P]),
        }
        for name, (res, args) in sigs.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _LIBS[variant] = lib
    return _LIBS[variant]


def dtype_of(variant: str):
    return np.float64 if variant == "f64" else np.float32


def _p(a: np.ndarray | None):
    return None if a is None else a.ctypes.data


class Ops:
    """Per-layer oracle functions on numpy arrays of the variant's dtype."""

    def __init__(self, variant: str = "f64"):
        self.lib = _lib(variant)
        self.dt = dtype_of(variant)

    def _c(self, a):
        return np.ascontiguousarray(a, dtype=self.dt)

    def gelu(self, x):
        x = self._c(x)
        out = np.empty_like(x)
        self.lib.or_gelu_forward(_p(out), _p(x), x.size)
        return out

    def gelu_backward(self, x, dout):
        x, dout = self._c(x), self._c(dout)
        dx = np.zeros_like(x)
        self.lib.or_gelu_backward(_p(dx), _p(x), _p(dout), x.size)
        return dx

    def softmax(self, logits):
        logits = self._c(logits)
        V = logits.shape[-1]
        rows = logits.size // V
        probs = np.empty_like(logits)
        self.lib.or_softmax_forward(_p(probs), _p(logits), 1, rows, V)
        return probs

    def layernorm(self, x, w, b):
        x, w, b = self._c(x), self._c(w), self._c(b)
        C = x.shape[-1]
        rows = x.size // C
        out = np.empty_like(x)
        mean = np.empty(rows, self.dt)
        rstd = np.empty(rows, self.dt)
        self.lib.or_layernorm_forward(_p(out), _p(mean), _p(rstd), _p(x), _p(w), _p(b), 1, rows, C)
        return out, mean, rstd

    def layernorm_backward(self, dout, x, w, mean, rstd):
        dout, x, w = self._c(dout), self._c(x), self._c(w)
        C = x.shape[-1]
        rows = x.size // C
        dx = np.zeros_like(x)
        dw = np.zeros(C, self.dt)
        db = np.zeros(C, self.dt)
        self.lib.or_layernorm_backward(_p(dx), _p(dw), _p(db), _p(dout), _p(x), _p(w),
                                       _p(self._c(mean)), _p(self._c(rstd)), 1, rows, C)
        return dx, dw, db

    def rmsnorm(self, x, w):
        """microGPT's RMSNorm: out = x / sqrt(mean(x^2) + 1e-5) * w; returns (out, rstd)."""
        x, w = self._c(x), self._c(w)
        C = x.shape[-1]
        rows = x.size // C
        out = np.empty_like(x)
        rstd = np.empty(rows, self.dt)
        self.lib.or_rmsnorm_forward(_p(out), _p(rstd), _p(x), _p(w), 1, rows, C)
        return out, rstd

    def rmsnorm_backward(self, dout, x, w, rstd):
        dout, x, w = self._c(dout), self._c(x), self._c(w)
        C = x.shape[-1]
        rows = x.size // C
        dx = np.zeros_like(x)
        dw = np.zeros(C, self.dt)
        self.lib.or_rmsnorm_backward(_p(dx), _p(dw), _p(dout), _p(x), _p(w), _p(self._c(rstd)), 1, rows, C)
        return dx, dw

    def matmul(self, x, W, bias=None):
        x, W = self._c(x), self._c(W)
        C = x.shape[-1]
        OC = W.shape[0]
        rows = x.size // C
        out = np.empty(x.shape[:-1] + (OC,), self.dt)
        self.lib.or_matmul_forward(_p(out), _p(x), _p(W), _p(None if bias is None else self._c(bias)),
                                   1, rows, C, OC)
        return out

    def matmul_backward(self, dout, x, W, with_bias=True):
        dout, x, W = self._c(dout), self._c(x), self._c(W)
        C = x.shape[-1]
        OC = W.shape[0]
        rows = x.size // C
        dx = np.zeros_like(x)
        dW = np.zeros_like(W)
        db = np.zeros(OC, self.dt) if with_bias else None
        self.lib.or_matmul_backward(_p(dx), _p(dW), _p(db), _p(dout), _p(x), _p(W), 1, rows, C, OC)
        return dx, dW, db

    def attention(self, qkv, NH):
        qkv = self._c(qkv)
        B, T, C3 = qkv.shape
        C = C3 // 3
        out = np.empty((B, T, C), self.dt)
        pre = np.zeros((B, NH, T, T), self.dt)
        att = np.zeros((B, NH, T, T), self.dt)
        self.lib.or_attention_forward(_p(out), _p(pre), _p(att), _p(qkv), B, T, C, NH)
        return out, pre, att

    def attention_backward(self, dout, qkv, att, NH):
        dout, qkv, att = self._c(dout), self._c(qkv), self._c(att)
        B, T, C3 = qkv.shape
        C = C3 // 3
        dqkv = np.zeros_like(qkv)
        dpre = np.zeros((B, NH, T, T), self.dt)
        datt = np.zeros((B, NH, T, T), self.dt)
        self.lib.or_attention_backward(_p(dqkv), _p(dpre), _p(datt), _p(dout), _p(qkv), _p(att),
                                       B, T, C, NH)
        return dqkv

    def encoder(self, tokens, wte, wpe):
        tokens = np.ascontiguousarray(tokens, np.int32)
        wte, wpe = self._c(wte), self._c(wpe)
        B, T = tokens.shape
        C = wte.shape[1]
        out = np.empty((B, T, C), self.dt)
        self.lib.or_encoder_forward(_p(out), _p(tokens), _p(wte), _p(wpe), B, T, C)
        return out

    def encoder_backward(self, dout, tokens, V, maxT):
        tokens = np.ascontiguousarray(tokens, np.int32)
        dout = self._c(dout)
        B, T, C = dout.shape
        dwte = np.zeros((V, C), self.dt)
        dwpe = np.zeros((maxT, C), self.dt)
        self.lib.or_encoder_backward(_p(dwte), _p(dwpe), _p(dout), _p(tokens), B, T, C)
        return dwte, dwpe

    def cross_entropy(self, logits, targets):
        """Mean loss, per-row losses and dlogits for dloss = 1/rows (llm.c 1.13-1.15)."""
        logits = self._c(logits)
        targets = np.ascontiguousarray(targets, np.int32).reshape(-1)
        V = logits.shape[-1]
        rows = logits.size // V
        probs = np.empty_like(logits)
        self.lib.or_softmax_forward(_p(probs), _p(logits), 1, rows, V)
        losses = np.empty(rows, self.dt)
        self.lib.or_crossentropy_forward(_p(losses), _p(probs), _p(targets), 1, rows, V)
        dl = np.full(rows, 1.0 / rows, self.dt)
        dlogits = np.zeros_like(logits)
        self.lib.or_crossentropy_softmax_backward(_p(dlogits), _p(dl), _p(probs), _p(targets), 1, rows, V)
        return losses.mean(), losses, dlogits

    def sample_mult(self, probs, coin):
        """llm.c section 1.35: first index whose cumulative probability exceeds coin."""
        probs = self._c(probs)
        return int(self.lib.or_sample_mult(_p(probs), probs.size, float(coin)))

    def adamw(self, p, g, m, v, lr, b1, b2, eps, wd, t):
        """Returns updated (p, m, v); inputs are not modified."""
        p, g, m, v = (self._c(a).copy() for a in (p, g, m, v))
        rc = self.lib.or_adamw(_p(p), _p(g), _p(m), _p(v), p.size, lr, b1, b2, eps, wd, t)
        if rc != 0:
            raise ValueError("or_adamw: t must be >= 1")
        return p, m, v


class Model:
    """The oracle's whole-model step (llm.c sections 1.22-1.27).

    norm: "layernorm" (GPT-2) or "rmsnorm" (the microGPT variant: every LayerNorm
    replaced by RMSNorm with gain, the shift tensors carried unused)."""

    NORMS = {"layernorm": 0, "rmsnorm": 1}

    def __init__(self, L, C, NH, V, maxT, variant: str = "f64", norm: str = "layernorm"):
        self.lib = _lib(variant)
        self.dt = dtype_of(variant)
        self.L, self.C, self.NH, self.V, self.maxT = L, C, NH, V, maxT
        self.norm = norm
        self.h = self.lib.or_build_ex(L, C, NH, V, maxT, self.NORMS[norm])
        if not self.h:
            raise ValueError("or_build failed")
        self.n = self.lib.or_num_params(self.h)
        self.B = self.T = None

    def __del__(self):
        if getattr(self, "h", None):
            self.lib.or_free(self.h)
            self.h = None

    def set_params(self, flat):
        flat = np.ascontiguousarray(flat, dtype=self.dt)
        assert flat.size == self.n
        self.lib.or_set_params(self.h, _p(flat))

    def params(self):
        out = np.empty(self.n, self.dt)
        self.lib.or_get_params(self.h, _p(out))
        return out

    def grads(self):
        out = np.empty(self.n, self.dt)
        if self.lib.or_get_grads(self.h, _p(out)) != 0:
            raise RuntimeError("no gradients yet")
        return out

    def opt_state(self):
        m = np.empty(self.n, self.dt)
        v = np.empty(self.n, self.dt)
        if self.lib.or_get_opt_state(self.h, _p(m), _p(v)) != 0:
            raise RuntimeError("no optimizer state yet")
        return m, v

    def forward(self, inputs, targets=None):
        inputs = np.ascontiguousarray(inputs, np.int32)
        B, T = inputs.shape
        tg = None if targets is None else np.ascontiguousarray(targets, np.int32)
        loss = (ct.c_double if self.dt == np.float64 else ct.c_float)()
        rc = self.lib.or_forward(self.h, _p(inputs), _p(tg), B, T, ct.addressof(loss))
        if rc != 0:
            raise ValueError(f"or_forward failed with code {rc}")
        self.B, self.T = B, T
        return float(loss.value)

    def logits(self):
        out = np.empty((self.B, self.T, self.V), self.dt)
        if self.lib.or_get_logits(self.h, _p(out)) != 0:
            raise RuntimeError("no forward yet")
        return out

    def losses(self):
        out = np.empty((self.B, self.T), self.dt)
        if self.lib.or_get_losses(self.h, _p(out)) != 0:
            raise RuntimeError("no forward with targets yet")
        return out

    def dencoded(self):
        out = np.empty((self.B, self.T, self.C), self.dt)
        if self.lib.or_get_dencoded(self.h, _p(out)) != 0:
            raise RuntimeError("no backward yet")
        return out

    def zero_grad(self):
        self.lib.or_zero_grad(self.h)

    def backward(self, zero_first: bool = True):
        if zero_first:
            self.zero_grad()
        rc = self.lib.or_backward(self.h)
        if rc != 0:
            raise RuntimeError(f"or_backward failed with code {rc}")

    def update(self, lr, b1, b2, eps, wd, t):
        rc = self.lib.or_update(self.h, lr, b1, b2, eps, wd, t)
        if rc != 0:
            raise RuntimeError(f"or_update failed with code {rc}")

    def release_acts(self):
        """Forget the activation shape so the next forward may use another (B, T)."""
        self.lib.or_release_acts(self.h)
        self.B = self.T = None

    def generate(self, prompt, n_new, temperature=0.0, coins=None):
        """picoGPT's generate: (B, n_new) new ids; greedy when temperature <= 0, else
        sample_mult over softmax(logits / temperature) with coins (B, n_new) in [0, 1)."""
        prompt = np.ascontiguousarray(prompt, np.int32)
        B, T0 = prompt.shape
        out = np.zeros((B, n_new), np.int32)
        c = None if coins is None else np.ascontiguousarray(coins, self.dt).reshape(B, n_new)
        if temperature > 0 and c is None:
            raise ValueError("sampling needs coins")
        rc = self.lib.or_generate(self.h, _p(prompt), B, T0, n_new, float(temperature), _p(c), _p(out))
        if rc != 0:
            raise ValueError(f"or_generate failed with code {rc}")
        self.B = self.T = None
        return out


def set_threads(n: int, variant: str = "f64") -> int:
    """Threads of the oracle's OpenMP loops from now on (n <= 0 keeps them); returns the
    count in force.  Results do not depend on it."""
    return int(_lib(variant).or_set_threads(int(n)))


def cpu_threads() -> int:
    v = os.environ.get("OMP_NUM_THREADS")
    return int(v) if v and v.isdigit() else (os.cpu_count() or 1)
