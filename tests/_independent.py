"""Independent statements of the GPT-2 step used to pin the CPU oracle.

Neither helper shares code with the oracle or with the CUDA library:

* ``picogpt_logits`` restates the forward the way the picoGPT article writes it
  (functions gpt2, transformer_block, mha with causal_mask, ffn, layer_norm,
  gelu, linear) in numpy float64, with the article's [in, out] weight layout,
  i.e. the transposes of the llm.c (out, in) layout.
* ``torch_loss_and_grads`` states the same model with PyTorch library routines
  (layer_norm, the tanh GELU, masked softmax, cross_entropy) in float64 and
  lets autograd produce the gradients; with norm="rmsnorm" it states the microGPT
  variant with torch's rms_norm.
"""
from __future__ import annotations

import math

import numpy as np

from gpt_train_step_arena_b300.synth import PARAM_NAMES, param_sizes


def unflatten(flat, L, C, V, maxT):
    out, off = {}, 0
    shapes = {
        "wte": (V, C), "wpe": (maxT, C), "ln1w": (L, C), "ln1b": (L, C), "qkvw": (L, 3 * C, C),
        "qkvb": (L, 3 * C), "attprojw": (L, C, C), "attprojb": (L, C), "ln2w": (L, C),
        "ln2b": (L, C), "fcw": (L, 4 * C, C), "fcb": (L, 4 * C), "fcprojw": (L, C, 4 * C),
        "fcprojb": (L, C), "lnfw": (C,), "lnfb": (C,),
    }
    for name, n in zip(PARAM_NAMES, param_sizes(L, C, V, maxT)):
        out[name] = flat[off:off + n].reshape(shapes[name])
        off += n
    return out


# ---- picoGPT article, restated in numpy float64 ----------------------------

def _gelu(x):
    return 0.5 * x * (1 + np.tanh(np.sqrt(2 / np.pi) * (x + 0.044715 * x ** 3)))


def _softmax(x):
    e = np.exp(x - np.max(x, axis=-1, keepdims=True))
    return e / np.sum(e, axis=-1, keepdims=True)


def _layer_norm(x, g, b, eps=1e-5):
    mu = np.mean(x, axis=-1, keepdims=True)
    var = np.var(x, axis=-1, keepdims=True)
    return g * (x - mu) / np.sqrt(var + eps) + b


def _linear(x, w, b):  # w is [in, out]
    return x @ w + b


def _attention(q, k, v, mask):
    return _softmax(q @ k.T / np.sqrt(q.shape[-1]) + mask) @ v


def _mha(x, w_attn, b_attn, w_proj, b_proj, n_head):
    x = _linear(x, w_attn, b_attn)
    qkv = np.split(x, 3, axis=-1)
    heads = [np.split(t, n_head, axis=-1) for t in qkv]
    mask = (1 - np.tri(x.shape[0])) * -1e10
    outs = [_attention(q, k, v, mask) for q, k, v in zip(*heads)]
    return _linear(np.hstack(outs), w_proj, b_proj)


def _rms_norm(x, g, b, eps=1e-5):  # b unused: RMSNorm has no shift
    return g * x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)


def picogpt_logits(flat, tokens, L, C, NH, V, maxT, norm="layernorm"):
    """(B, T, V) logits from the picoGPT formulation, one sequence at a time; norm="rmsnorm"
    puts root-mean-square normalisation (gain, no shift) in place of every layer_norm."""
    nf = _rms_norm if norm == "rmsnorm" else _layer_norm
    P = unflatten(np.asarray(flat, np.float64), L, C, V, maxT)
    res = []
    for seq in np.asarray(tokens):
        x = P["wte"][seq] + P["wpe"][np.arange(len(seq))]
        for l in range(L):
            h = nf(x, P["ln1w"][l], P["ln1b"][l])
            x = x + _mha(h, P["qkvw"][l].T, P["qkvb"][l], P["attprojw"][l].T, P["attprojb"][l], NH)
            h = nf(x, P["ln2w"][l], P["ln2b"][l])
            a = _gelu(_linear(h, P["fcw"][l].T, P["fcb"][l]))
            x = x + _linear(a, P["fcprojw"][l].T, P["fcprojb"][l])
        x = nf(x, P["lnfw"], P["lnfb"])
        res.append(x @ P["wte"].T)
    return np.stack(res)


# ---- PyTorch library routines + autograd, float64 ---------------------------

def torch_loss_and_grads(flat, tokens, targets, L, C, NH, V, maxT, norm="layernorm"):
    """norm="rmsnorm" states the microGPT variant: torch's rms_norm (eps 1e-5, gain =
    the ln*w tensors) in place of every layer_norm; the ln*b tensors are not used."""
    import torch
    import torch.nn.functional as F

    def normalise(x, w, b):
        if norm == "rmsnorm":
            return F.rms_norm(x, (C,), w, eps=1e-5)
        return F.layer_norm(x, (C,), w, b, eps=1e-5)

    p = torch.tensor(np.asarray(flat, np.float64), requires_grad=True)
    P = unflatten(p, L, C, V, maxT)
    tok = torch.tensor(np.asarray(tokens, np.int64))
    tgt = torch.tensor(np.asarray(targets, np.int64))
    B, T = tok.shape
    hs = C // NH
    x = P["wte"][tok] + P["wpe"][:T].unsqueeze(0)
    causal = torch.ones(T, T, dtype=torch.bool).tril()
    for l in range(L):
        h = normalise(x, P["ln1w"][l], P["ln1b"][l])
        qkv = F.linear(h, P["qkvw"][l], P["qkvb"][l])
        q, k, v = qkv.split(C, dim=-1)
        q = q.view(B, T, NH, hs).transpose(1, 2)
        k = k.view(B, T, NH, hs).transpose(1, 2)
        v = v.view(B, T, NH, hs).transpose(1, 2)
        s = (q @ k.transpose(-1, -2)) / math.sqrt(hs)
        s = s.masked_fill(~causal, float("-inf"))
        y = (torch.softmax(s, dim=-1) @ v).transpose(1, 2).reshape(B, T, C)
        x = x + F.linear(y, P["attprojw"][l], P["attprojb"][l])
        h = normalise(x, P["ln2w"][l], P["ln2b"][l])
        a = F.gelu(F.linear(h, P["fcw"][l], P["fcb"][l]), approximate="tanh")
        x = x + F.linear(a, P["fcprojw"][l], P["fcprojb"][l])
    x = normalise(x, P["lnfw"], P["lnfb"])
    logits = x @ P["wte"].T
    loss = F.cross_entropy(logits.reshape(B * T, V), tgt.reshape(B * T))
    loss.backward()
    return float(loss.detach()), p.grad.numpy().copy(), logits.detach().numpy()
