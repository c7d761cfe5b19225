"""Python face of the C ABI: the GPT2 handle with the same calls as include/gpt2.h.

Marshalling only (numpy arrays and torch tensors to pointers).  Every step of the
training step runs in the CUDA library.
"""
from __future__ import annotations

import ctypes as ct

import numpy as np

from . import _native as N


class GPT2Error(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{N.STATUS_NAMES.get(code, code)}: {msg}")
        self.code = code


def _ptr(a):
    if a is None:
        return None
    if isinstance(a, np.ndarray):
        return a.ctypes.data
    return a.data_ptr()  # torch tensor


class GPT2:
    """One model on the current CUDA device (gpt2_build_norm).

    norm: "layernorm" (GPT-2) or "rmsnorm" (the microGPT variant)."""

    def __init__(self, L: int, C: int, H: int, V: int, maxT: int, precision: str = "bf16",
                 norm: str = "layernorm"):
        prec = {"bf16": N.GPT2_BF16, "fp32": N.GPT2_FP32, "tf32": N.GPT2_TF32}[precision]
        nk = {"layernorm": N.GPT2_LAYERNORM, "rmsnorm": N.GPT2_RMSNORM}[norm]
        st = ct.c_int(0)
        h = N.lib.gpt2_build_norm(L, C, H, V, maxT, prec, nk, ct.byref(st))
        if not h:
            raise GPT2Error(st.value, N.lib.gpt2_last_build_error().decode())
        self.h = h
        self.L, self.C, self.H, self.V, self.maxT, self.precision = L, C, H, V, maxT, precision
        self.norm = norm
        self.n = N.lib.gpt2_num_params(h)
        self.Vp = N.lib.gpt2_padded_vocab(h)

    def close(self):
        if getattr(self, "h", None):
            N.lib.gpt2_free(self.h)
            self.h = None

    def __del__(self):
        self.close()

    # -- errors
    def _check(self, rc: int):
        if rc != N.GPT2_OK:
            raise GPT2Error(rc, N.lib.gpt2_last_error(self.h).decode())

    def last_status(self) -> int:
        return N.lib.gpt2_last_status(self.h)

    # -- parameters
    def set_params(self, flat: np.ndarray):
        flat = np.ascontiguousarray(flat, dtype=np.float32)
        self._check(N.lib.gpt2_set_params(self.h, _ptr(flat), flat.size))

    def init_params(self, seed: int = 42):
        """The seeded initial parameters, drawn on the device (gpt2_init_params)."""
        self._check(N.lib.gpt2_init_params(self.h, seed))

    def params(self) -> np.ndarray:
        out = np.empty(self.n, np.float32)
        self._check(N.lib.gpt2_get_params(self.h, _ptr(out), out.size))
        return out

    def grads(self) -> np.ndarray:
        out = np.empty(self.n, np.float32)
        self._check(N.lib.gpt2_get_grads(self.h, _ptr(out), out.size))
        return out

    def opt_state(self):
        m = np.empty(self.n, np.float32)
        v = np.empty(self.n, np.float32)
        self._check(N.lib.gpt2_get_opt_state(self.h, _ptr(m), _ptr(v), self.n))
        return m, v

    # -- step
    def forward(self, tokens: np.ndarray, targets: np.ndarray | None = None) -> float:
        tokens = np.ascontiguousarray(tokens, dtype=np.int32)
        tg = None if targets is None else np.ascontiguousarray(targets, dtype=np.int32)
        B, T = tokens.shape
        loss = N.lib.gpt2_forward(self.h, _ptr(tokens), _ptr(tg), B, T)
        if np.isnan(loss):
            self._check(self.last_status() or N.GPT2_ERR_NONFINITE)
        return float(loss)

    def forward_async(self, tokens, targets=None, B=None, T=None, device: bool = False):
        """tokens/targets: numpy (host) or torch tensors (host pinned or device)."""
        if B is None:
            B, T = tokens.shape
        where = N.GPT2_DEVICE if device else N.GPT2_HOST
        self._check(N.lib.gpt2_forward_async(self.h, _ptr(tokens), _ptr(targets), B, T, where))

    def read_loss(self) -> float:
        out = ct.c_float(0)
        self._check(N.lib.gpt2_read_loss(self.h, ct.byref(out)))
        return float(out.value)

    def backward(self):
        self._check(N.lib.gpt2_backward(self.h))

    def zero_grad(self):
        self._check(N.lib.gpt2_zero_grad(self.h))

    def update(self, lr, b1, b2, eps, wd, t):
        self._check(N.lib.gpt2_update(self.h, lr, b1, b2, eps, wd, t))

    # -- accessors
    def losses(self, B: int, T: int) -> np.ndarray:
        out = np.empty((B, T), np.float32)
        self._check(N.lib.gpt2_get_losses(self.h, _ptr(out), out.size))
        return out

    def logits(self, B: int, T: int) -> np.ndarray:
        out = np.empty((B, T, self.V), np.float32)
        self._check(N.lib.gpt2_get_logits(self.h, _ptr(out), out.size))
        return out

    # -- generation
    def generate(self, prompt, n_new: int, temperature: float = 0.0, coins=None) -> np.ndarray:
        """(B, n_new) new ids after the (B, T0) int32 prompt: greedy when temperature <= 0,
        else sampled with the caller's coins (B, n_new) in [0, 1)."""
        prompt = np.ascontiguousarray(prompt, np.int32)
        B, T0 = prompt.shape
        out = np.zeros((B, n_new), np.int32)
        c = None if coins is None else np.ascontiguousarray(coins, np.float32).reshape(B, n_new)
        self._check(N.lib.gpt2_generate(self.h, _ptr(prompt), B, T0, n_new, float(temperature),
                                        None if c is None else _ptr(c), _ptr(out)))
        return out

    def gen_logits(self, B: int) -> np.ndarray:
        """(B, V) logits of the last generation step."""
        out = np.empty((B, self.V), np.float32)
        self._check(N.lib.gpt2_get_gen_logits(self.h, _ptr(out), out.size))
        return out

    def ids(self, B: int, T: int):
        tok = np.empty((B, T), np.int32)
        tgt = np.empty((B, T), np.int32)
        self._check(N.lib.gpt2_get_ids(self.h, _ptr(tok), _ptr(tgt), tok.size))
        return tok, tgt

    def set_stream(self, stream_ptr: int | None):
        self._check(N.lib.gpt2_set_stream(self.h, stream_ptr))

    def sync(self):
        self._check(N.lib.gpt2_sync(self.h))

    def profile_enable(self, on: bool = True):
        self._check(N.lib.gpt2_profile_enable(self.h, 1 if on else 0))

    def profile_reset(self):
        self._check(N.lib.gpt2_profile_reset(self.h))

    def profile_read(self) -> dict:
        """{class: (ms, work, calls)} accumulated since the last reset."""
        out = {}
        for k, name in enumerate(N.KERNEL_CLASSES):
            ms, work, calls = ct.c_double(), ct.c_double(), ct.c_uint64()
            self._check(N.lib.gpt2_profile_read(self.h, k, ct.byref(ms), ct.byref(work), ct.byref(calls)))
            out[name] = (ms.value, work.value, int(calls.value))
        return out

    def kernel_launches(self) -> int:
        return int(N.lib.gpt2_kernel_launches(self.h))

    def device_bytes(self) -> int:
        return int(N.lib.gpt2_device_bytes(self.h))
