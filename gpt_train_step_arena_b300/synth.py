"""Seeded synthetic inputs for the GPT-2 train step: token streams and initial weights.

This module only draws random numbers and lays them out.  It holds none of the
training step's arithmetic, so both the CPU oracle (tests) and the CUDA library
(tests, bench) can be fed from it without sharing any compute code.

Generator: xorshift64* as printed in the llm.c annotated listing (page
"llm.c 的中文注解-20240421", section 1.33 random_u32) with the float mapping of
section 1.34 random_f32 (top 24 bits / 2^24).  To make multi-million draws fast in
numpy, ``LANES`` independent xorshift64* streams run side by side; lane ``j`` is
seeded with splitmix64(seed + j) (never zero), and draw ``i`` of a request comes
from lane ``i % LANES``, round ``i // LANES``.  The result is fully determined by
the seed.

Workload recipe (the stand-in for the text datasets the pages train on):
  * Zipf(s) token ids over the real vocabulary: P(k) proportional to (k+1)^-s,
    sampled with the rule of section 1.35 sample_mult (first k whose CDF exceeds
    the coin, else the last id) on a float64 CDF.
  * uniform ids (``u32 % V``) for the char-level case.
  * targets are the same stream shifted by one (section 1.30 dataloader_next_batch
    reads B*T+1 tokens and takes targets = inputs + 1; picoGPT's lm_loss uses
    ``inputs[1:]``).
  * weights N(0, 0.02) by Box-Muller on random_f32 pairs; the two residual
    projections (attproj, fcproj) use 0.02/sqrt(2L); biases 0; LayerNorm gain 1
    and shift 0.
"""
from __future__ import annotations

import math

import numpy as np

LANES = 1 << 16
_MUL = np.uint64(0x2545F4914F6CDD1D)


def _splitmix64(x: np.ndarray) -> np.ndarray:
    """splitmix64 finaliser (Steele, Lea, Flood 2014), used only to seed lanes."""
    with np.errstate(over="ignore"):
        z = (x + np.uint64(0x9E3779B97F4A7C15)).astype(np.uint64)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        z = z ^ (z >> np.uint64(31))
    z[z == 0] = np.uint64(0x9E3779B97F4A7C15)
    return z


class XorShiftStreams:
    """``LANES`` parallel xorshift64* generators (llm.c section 1.33)."""

    def __init__(self, seed: int, lanes: int = LANES):
        base = np.uint64(seed & 0xFFFFFFFFFFFFFFFF)
        with np.errstate(over="ignore"):
            idx = np.arange(lanes, dtype=np.uint64) + base
        self.state = _splitmix64(idx)
        self.lanes = lanes

    def _step(self) -> np.ndarray:
        s = self.state
        with np.errstate(over="ignore"):
            s ^= s >> np.uint64(12)
            s ^= s << np.uint64(25)
            s ^= s >> np.uint64(27)
            out = (s * _MUL) >> np.uint64(32)
        return out.astype(np.uint32)

    def u32(self, n: int) -> np.ndarray:
        rounds = (n + self.lanes - 1) // self.lanes
        out = np.empty((rounds, self.lanes), dtype=np.uint32)
        for r in range(rounds):
            out[r] = self._step()
        return out.reshape(-1)[:n]

    def f32(self, n: int) -> np.ndarray:
        """random_f32 of section 1.34: (u32 >> 8) / 2^24, in [0, 1)."""
        return ((self.u32(n) >> np.uint32(8)).astype(np.float32) / np.float32(16777216.0))

    def normal(self, n: int, std: float) -> np.ndarray:
        """Box-Muller pairs from random_f32; u1 is kept away from 0."""
        m = (n + 1) // 2
        u = self.f32(2 * m).astype(np.float64)
        u1 = np.maximum(u[0::2], 1e-7)
        u2 = u[1::2]
        r = np.sqrt(-2.0 * np.log(u1))
        z = np.empty(2 * m, dtype=np.float64)
        z[0::2] = r * np.cos(2.0 * math.pi * u2)
        z[1::2] = r * np.sin(2.0 * math.pi * u2)
        return (z[:n] * std).astype(np.float32)


def param_sizes(L: int, C: int, V: int, maxT: int) -> list[int]:
    """Element counts of the 16 parameter tensors in the order of llm.c section 1.16
    (wte, wpe, ln1w, ln1b, qkvw, qkvb, attprojw, attprojb, ln2w, ln2b, fcw, fcb,
    fcprojw, fcprojb, lnfw, lnfb) with the sizes of section 1.22."""
    return [V * C, maxT * C, L * C, L * C, L * 3 * C * C, L * 3 * C, L * C * C, L * C,
            L * C, L * C, L * 4 * C * C, L * 4 * C, L * 4 * C * C, L * C, C, C]


PARAM_NAMES = ["wte", "wpe", "ln1w", "ln1b", "qkvw", "qkvb", "attprojw", "attprojb",
               "ln2w", "ln2b", "fcw", "fcb", "fcprojw", "fcprojb", "lnfw", "lnfb"]


def split_params(flat: np.ndarray, L: int, C: int, V: int, maxT: int) -> dict:
    """Views of a flat parameter-ordered array, one per tensor name."""
    out, off = {}, 0
    for name, n in zip(PARAM_NAMES, param_sizes(L, C, V, maxT)):
        out[name] = flat[off:off + n]
        off += n
    assert off == flat.size, (off, flat.size)
    return out


def init_params(L: int, C: int, V: int, maxT: int, seed: int = 42, std: float = 0.02) -> np.ndarray:
    """Flat float32 initial parameters in the section-1.16 order (real vocabulary V)."""
    sizes = param_sizes(L, C, V, maxT)
    rng = XorShiftStreams(seed)
    proj_std = std / math.sqrt(2.0 * L)
    kinds = ["n", "n", "1", "0", "n", "0", "p", "0", "1", "0", "n", "0", "p", "0", "1", "0"]
    parts = []
    for n, k in zip(sizes, kinds):
        if k == "n":
            parts.append(rng.normal(n, std))
        elif k == "p":
            parts.append(rng.normal(n, proj_std))
        elif k == "1":
            parts.append(np.ones(n, dtype=np.float32))
        else:
            parts.append(np.zeros(n, dtype=np.float32))
    return np.concatenate(parts)


def zipf_stream(V: int, n: int, s: float = 1.1, seed: int = 1337) -> np.ndarray:
    """n int32 token ids, P(k) ~ (k+1)^-s, sampled by the sample_mult rule."""
    k = np.arange(1, V + 1, dtype=np.float64)
    w = k ** (-s)
    cdf = np.cumsum(w / w.sum())
    coins = XorShiftStreams(seed).f32(n).astype(np.float64)
    ids = np.searchsorted(cdf, coins, side="right")
    return np.minimum(ids, V - 1).astype(np.int32)


def uniform_stream(V: int, n: int, seed: int = 1337) -> np.ndarray:
    return (XorShiftStreams(seed).u32(n) % np.uint32(V)).astype(np.int32)


def batch(stream: np.ndarray, step: int, B: int, T: int):
    """(inputs, targets) of shape (B, T) for the given step; targets = inputs + 1."""
    base = step * B * T
    need = base + B * T + 1
    if stream.size < need:
        raise ValueError(f"stream of {stream.size} tokens too short for step {step} (needs {need})")
    inp = np.ascontiguousarray(stream[base:base + B * T].reshape(B, T))
    tgt = np.ascontiguousarray(stream[base + 1:base + B * T + 1].reshape(B, T))
    return inp, tgt


# Named workloads (shapes of the GPT-2 training-step configurations).
WORKLOADS = {
    "tiny": dict(L=2, C=64, NH=4, V=512, maxT=32, B=4, T=32, dist="zipf",
                 lr=3e-4, b1=0.9, b2=0.999, eps=1e-8, wd=0.0, steps=1),
    "char": dict(L=1, C=16, NH=4, V=27, maxT=16, B=32, T=16, dist="uniform",
                 lr=1e-2, b1=0.9, b2=0.999, eps=1e-8, wd=0.0, steps=50),
    "gpt2_124m_small": dict(L=12, C=768, NH=12, V=50257, maxT=1024, B=4, T=64, dist="zipf",
                            lr=3e-4, b1=0.9, b2=0.999, eps=1e-8, wd=0.0, steps=1),
    "gpt2_124m": dict(L=12, C=768, NH=12, V=50257, maxT=1024, B=32, T=1024, dist="zipf",
                      lr=6e-4, b1=0.9, b2=0.999, eps=1e-8, wd=0.1, steps=25),
    "gpt2_350m": dict(L=24, C=1024, NH=16, V=50257, maxT=1024, B=16, T=1024, dist="zipf",
                      lr=6e-4, b1=0.9, b2=0.999, eps=1e-8, wd=0.0, steps=25),
}


def token_stream(cfg: dict, steps: int | None = None, seed: int = 1337) -> np.ndarray:
    steps = cfg["steps"] if steps is None else steps
    n = steps * cfg["B"] * cfg["T"] + 1
    if cfg["dist"] == "zipf":
        return zipf_stream(cfg["V"], n, seed=seed)
    return uniform_stream(cfg["V"], n, seed=seed)
