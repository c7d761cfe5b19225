"""Pins of the CPU oracle against what the pages and mathematics fix.

Each test ties one part of the oracle to something other than itself: worked
values printed on the picoGPT article page, closed forms, library routines
(numpy/scipy/PyTorch), brute-force finite differences, and the invariances the
llm.c listing states (nothing mixes batch rows; attention only looks back).
"""
import math
import os

import numpy as np
import pytest

from gpt_train_step_arena_b300 import synth
from oracle.oracle import Model, Ops

from ._independent import picogpt_logits, torch_loss_and_grads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "picogpt_worked_examples.txt")


def _golden():
    rows = {}
    for line in open(GOLDEN, encoding="utf-8"):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        name, inp, out = (s.strip() for s in line.split("|"))
        parse = lambda s: np.array([[float(v) for v in r.split()] for r in s.split(";")])
        rows[name] = (parse(inp), parse(out))
    return rows


def _printed_close(got, printed):
    # The page prints 5 significant digits: allow half a unit in the last printed place
    # (plus a hair for the page's own rounding).
    for g, p in zip(np.ravel(got), np.ravel(printed)):
        s = f"{p:.5g}"
        decimals = len(s.split(".")[1]) if "." in s else 0
        assert abs(g - p) <= 0.5 * 10 ** (-decimals) + 1e-12, (g, p)


ops = Ops("f64")


# ---------------------------------------------------------------- worked values

def test_gelu_worked_example():
    x, want = _golden()["gelu"]
    _printed_close(ops.gelu(x), want)


def test_softmax_worked_example_and_rows_sum_to_one():
    x, want = _golden()["softmax"]
    p = ops.softmax(x)
    _printed_close(p, want)
    rng = np.random.default_rng(0)
    z = rng.normal(scale=5.0, size=(64, 301))
    assert np.allclose(ops.softmax(z).sum(-1), 1.0, atol=1e-12)


def test_layernorm_worked_example_and_moments():
    x, want = _golden()["layernorm"]
    out, mean, rstd = ops.layernorm(x, np.ones(3), np.zeros(3))
    _printed_close(out, want)
    _, var_printed = _golden()["layernorm_var"]
    _printed_close(out.var(-1), var_printed)
    # closed form: with unit gain and zero shift every row has mean 0 and
    # variance v / (v + eps) where v is the row's biased input variance.
    rng = np.random.default_rng(1)
    z = rng.normal(size=(32, 97)) * 3 + 1
    o, m, r = ops.layernorm(z, np.ones(97), np.zeros(97))
    v = z.var(-1)
    assert np.allclose(o.mean(-1), 0, atol=1e-12)
    assert np.allclose(o.var(-1), v / (v + 1e-5), rtol=1e-12)
    assert np.allclose(m, z.mean(-1), rtol=1e-13)
    assert np.allclose(r, 1 / np.sqrt(v + 1e-5), rtol=1e-13)


# ---------------------------------------------------------------- library routines

def test_matmul_matches_numpy():
    rng = np.random.default_rng(2)
    x = rng.normal(size=(3, 5, 17))
    W = rng.normal(size=(11, 17))
    b = rng.normal(size=11)
    assert np.allclose(ops.matmul(x, W, b), x @ W.T + b, rtol=1e-13, atol=1e-13)
    assert np.allclose(ops.matmul(x, W), x @ W.T, rtol=1e-13, atol=1e-13)
    dy = rng.normal(size=(3, 5, 11))
    dx, dW, db = ops.matmul_backward(dy, x, W)
    assert np.allclose(dx, dy @ W, rtol=1e-12, atol=1e-12)
    assert np.allclose(dW, dy.reshape(-1, 11).T @ x.reshape(-1, 17), rtol=1e-12, atol=1e-12)
    assert np.allclose(db, dy.reshape(-1, 11).sum(0), rtol=1e-12, atol=1e-12)


def test_encoder_matches_indexing_and_scatter():
    rng = np.random.default_rng(3)
    V, C, maxT, B, T = 13, 8, 9, 3, 7
    wte, wpe = rng.normal(size=(V, C)), rng.normal(size=(maxT, C))
    tok = rng.integers(0, V, size=(B, T)).astype(np.int32)
    tok[0, :] = 4  # repeated ids exercise the scatter-add
    assert np.array_equal(ops.encoder(tok, wte, wpe), wte[tok] + wpe[np.arange(T)][None])
    d = rng.normal(size=(B, T, C))
    dwte, dwpe = ops.encoder_backward(d, tok, V, maxT)
    want_te = np.zeros((V, C))
    np.add.at(want_te, tok.reshape(-1), d.reshape(-1, C))
    want_pe = np.zeros((maxT, C))
    want_pe[:T] = d.sum(0)
    assert np.allclose(dwte, want_te, atol=1e-13)
    assert np.allclose(dwpe, want_pe, atol=1e-13)


def test_attention_loop_form_equals_dense_causal_form():
    """llm.c's explicit t2<=t loops must equal picoGPT's softmax(qk^T/sqrt(d)+mask)v."""
    rng = np.random.default_rng(4)
    B, T, C, NH = 2, 11, 24, 3
    hs = C // NH
    qkv = rng.normal(size=(B, T, 3 * C))
    out, pre, att = ops.attention(qkv, NH)
    mask = (1 - np.tri(T)) * -1e10
    for b in range(B):
        for h in range(NH):
            q = qkv[b, :, h * hs:(h + 1) * hs]
            k = qkv[b, :, C + h * hs:C + (h + 1) * hs]
            v = qkv[b, :, 2 * C + h * hs:2 * C + (h + 1) * hs]
            s = q @ k.T / np.sqrt(hs) + mask
            e = np.exp(s - s.max(-1, keepdims=True))
            a = e / e.sum(-1, keepdims=True)
            assert np.allclose(att[b, h], a, atol=1e-14)
            assert np.allclose(out[b, :, h * hs:(h + 1) * hs], a @ v, atol=1e-12)
    assert np.all(np.triu(att[0, 0], 1) == 0)


def test_cross_entropy_matches_logsumexp():
    from scipy.special import logsumexp
    rng = np.random.default_rng(5)
    logits = rng.normal(scale=3, size=(6, 40))
    tgt = rng.integers(0, 40, size=6)
    mean, losses, _ = ops.cross_entropy(logits, tgt)
    want = logsumexp(logits, axis=-1) - logits[np.arange(6), tgt]
    assert np.allclose(losses, want, rtol=1e-13)
    assert abs(mean - want.mean()) < 1e-13


# ---------------------------------------------------------------- finite differences (per layer)

def _fd(f, x, h=1e-6):
    g = np.zeros_like(x)
    flat, gf = x.reshape(-1), g.reshape(-1)
    for i in range(flat.size):
        old = flat[i]
        flat[i] = old + h
        fp = f()
        flat[i] = old - h
        fm = f()
        flat[i] = old
        gf[i] = (fp - fm) / (2 * h)
    return g


def test_gelu_backward_finite_difference():
    x = np.linspace(-6, 6, 49)
    d = np.ones_like(x)
    g = ops.gelu_backward(x, d)
    fd = np.array([(ops.gelu(np.array([v + 1e-6]))[0] - ops.gelu(np.array([v - 1e-6]))[0]) / 2e-6 for v in x])
    assert np.allclose(g, fd, atol=1e-8)


def test_layernorm_backward_finite_difference():
    rng = np.random.default_rng(6)
    x = rng.normal(size=(3, 10))
    w, b = rng.normal(size=10), rng.normal(size=10)
    dy = rng.normal(size=(3, 10))
    out, mean, rstd = ops.layernorm(x, w, b)
    dx, dw, db = ops.layernorm_backward(dy, x, w, mean, rstd)
    f = lambda: float((ops.layernorm(x, w, b)[0] * dy).sum())
    assert np.allclose(dx, _fd(f, x), atol=1e-8)
    assert np.allclose(dw, _fd(f, w), atol=1e-8)
    assert np.allclose(db, _fd(f, b), atol=1e-8)


def test_attention_backward_finite_difference():
    rng = np.random.default_rng(7)
    B, T, C, NH = 1, 5, 8, 2
    qkv = rng.normal(size=(B, T, 3 * C))
    dy = rng.normal(size=(B, T, C))
    _, _, att = ops.attention(qkv, NH)
    dqkv = ops.attention_backward(dy, qkv, att, NH)
    f = lambda: float((ops.attention(qkv, NH)[0] * dy).sum())
    assert np.allclose(dqkv, _fd(f, qkv), atol=1e-8)


def test_cross_entropy_backward_finite_difference():
    rng = np.random.default_rng(8)
    logits = rng.normal(size=(4, 9))
    tgt = rng.integers(0, 9, size=4)
    _, _, dl = ops.cross_entropy(logits, tgt)
    f = lambda: float(ops.cross_entropy(logits, tgt)[0])
    assert np.allclose(dl, _fd(f, logits), atol=1e-9)


# ---------------------------------------------------------------- AdamW closed forms

def test_adamw_first_step_closed_form():
    """At t=1 from zero moments, m_hat = g and v_hat = g^2, so the step is
    p - lr*(g/(|g|+eps) + wd*p)."""
    rng = np.random.default_rng(9)
    p, g = rng.normal(size=100), rng.normal(size=100)
    lr, eps, wd = 1e-3, 1e-8, 0.1
    p1, m1, v1 = ops.adamw(p, g, np.zeros(100), np.zeros(100), lr, 0.9, 0.999, eps, wd, 1)
    assert np.allclose(p1, p - lr * (g / (np.abs(g) + eps) + wd * p), rtol=1e-14, atol=1e-16)
    assert np.allclose(m1, 0.1 * g, rtol=1e-15)
    assert np.allclose(v1, 0.001 * g * g, rtol=1e-13)


def test_adamw_second_step_by_hand():
    p0, g1, g2 = 0.5, 0.2, -0.4
    lr, b1, b2, eps, wd = 0.01, 0.9, 0.999, 1e-8, 0.05
    p1, m1, v1 = ops.adamw(np.array([p0]), np.array([g1]), np.zeros(1), np.zeros(1), lr, b1, b2, eps, wd, 1)
    p2, m2, v2 = ops.adamw(p1, np.array([g2]), m1, v1, lr, b1, b2, eps, wd, 2)
    # by hand
    m = 0.1 * 0.2
    v = 0.001 * 0.04
    P1 = p0 - lr * ((m / 0.1) / (math.sqrt(v / 0.001) + eps) + wd * p0)
    m = 0.9 * m + 0.1 * (-0.4)
    v = 0.999 * v + 0.001 * 0.16
    mh = m / (1 - 0.9 ** 2)
    vh = v / (1 - 0.999 ** 2)
    P2 = P1 - lr * (mh / (math.sqrt(vh) + eps) + wd * P1)
    assert abs(p1[0] - P1) < 1e-15 and abs(p2[0] - P2) < 1e-15


def test_adamw_zero_grad_no_decay_is_identity():
    p = np.random.default_rng(10).normal(size=50)
    p1, _, _ = ops.adamw(p, np.zeros(50), np.zeros(50), np.zeros(50), 0.1, 0.9, 0.999, 1e-8, 0.0, 3)
    assert np.array_equal(p1, p)
    with pytest.raises(ValueError):
        ops.adamw(p, p, p, p, 0.1, 0.9, 0.999, 1e-8, 0.0, 0)


# ---------------------------------------------------------------- whole model

def test_parameter_count_gpt2_124m():
    # picoGPT hparams (n_vocab 50257, n_ctx 1024, n_embd 768, n_layer 12) with the
    # llm.c tensor sizes: 124,439,808 parameters.
    m = Model(12, 768, 12, 50257, 1024)
    assert m.n == 124_439_808
    assert sum(synth.param_sizes(12, 768, 50257, 1024)) == 124_439_808


def _cfg(name):
    c = synth.WORKLOADS[name]
    return c["L"], c["C"], c["NH"], c["V"], c["maxT"]


def test_forward_matches_picogpt_statement():
    L, C, NH, V, maxT = _cfg("tiny")
    params = synth.init_params(L, C, V, maxT, seed=11)
    tok = synth.zipf_stream(V, 2 * 12 + 1, seed=5)
    inp = tok[:24].reshape(2, 12)
    m = Model(L, C, NH, V, maxT)
    m.set_params(params)
    m.forward(inp)
    want = picogpt_logits(params, inp, L, C, NH, V, maxT)
    assert np.allclose(m.logits(), want, rtol=1e-11, atol=1e-12)


def test_whole_step_matches_torch_autograd():
    L, C, NH, V, maxT = _cfg("tiny")
    params = synth.init_params(L, C, V, maxT, seed=12)
    # make biases/LN non-trivial so every gradient term is exercised
    rng = np.random.default_rng(13)
    params = params + rng.normal(scale=0.02, size=params.size).astype(np.float32)
    stream = synth.zipf_stream(V, 4 * 32 + 1, seed=14)
    inp, tgt = synth.batch(stream, 0, 4, 32)
    m = Model(L, C, NH, V, maxT)
    m.set_params(params)
    loss = m.forward(inp, tgt)
    m.backward()
    tl, tg, tlog = torch_loss_and_grads(params, inp, tgt, L, C, NH, V, maxT)
    assert abs(loss - tl) <= 1e-12 * abs(tl)
    assert np.allclose(m.logits(), tlog, rtol=1e-10, atol=1e-12)
    g = m.grads()
    for name, a, b in zip(synth.PARAM_NAMES, np.split(g, np.cumsum(synth.param_sizes(L, C, V, maxT))[:-1]),
                          np.split(tg, np.cumsum(synth.param_sizes(L, C, V, maxT))[:-1])):
        err = np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)
        assert err < 1e-10, (name, err)


def _loss_fn(m, params, inp, tgt):
    def f():
        m.set_params(params)
        return m.forward(inp, tgt)
    return f


def test_whole_model_finite_difference_char_all_params():
    """Central differences in double on every parameter of the char-level model."""
    L, C, NH, V, maxT = _cfg("char")
    params = synth.init_params(L, C, V, maxT, seed=21).astype(np.float64)
    params += np.random.default_rng(22).normal(scale=0.05, size=params.size)
    stream = synth.uniform_stream(V, 4 * 16 + 1, seed=23)
    inp, tgt = synth.batch(stream, 0, 4, 16)
    m = Model(L, C, NH, V, maxT)
    f = _loss_fn(m, params, inp, tgt)
    f()
    m.backward()
    g = m.grads()
    fd = _fd(f, params, h=1e-6)
    # loss evaluations carry ~1e-15 rounding, i.e. ~1e-9 after dividing by 2h;
    # truncation is O(h^2).
    assert np.all(np.abs(fd - g) <= 1e-6 * np.abs(g) + 2e-9), np.max(np.abs(fd - g))


def test_whole_model_finite_difference_tiny_sampled():
    L, C, NH, V, maxT = _cfg("tiny")
    params = synth.init_params(L, C, V, maxT, seed=31).astype(np.float64)
    params += np.random.default_rng(32).normal(scale=0.02, size=params.size)
    stream = synth.zipf_stream(V, 2 * 16 + 1, seed=33)
    inp, tgt = synth.batch(stream, 0, 2, 16)
    m = Model(L, C, NH, V, maxT)
    m.set_params(params)
    m.forward(inp, tgt)
    m.backward()
    g = m.grads()
    rng = np.random.default_rng(34)
    offs = np.concatenate([[0], np.cumsum(synth.param_sizes(L, C, V, maxT))])
    idx = []
    for a, b in zip(offs[:-1], offs[1:]):
        idx += list(rng.choice(np.arange(a, b), size=min(24, b - a), replace=False))
    # include the rows of the tokens actually used so wte gradients are non-zero
    idx += [int(inp[0, 0]) * C + j for j in range(4)]
    for i in idx:
        old = params[i]
        params[i] = old + 1e-6
        m.set_params(params)
        lp = m.forward(inp, tgt)
        params[i] = old - 1e-6
        m.set_params(params)
        lm = m.forward(inp, tgt)
        params[i] = old
        fd = (lp - lm) / 2e-6
        assert abs(fd - g[i]) <= 1e-6 * abs(g[i]) + 2e-9, (i, fd, g[i])


def test_initial_loss_near_log_vocab_and_exact_special_case():
    L, C, NH, V, maxT = _cfg("tiny")
    params = synth.init_params(L, C, V, maxT, seed=42)
    stream = synth.zipf_stream(V, 4 * 32 + 1)
    inp, tgt = synth.batch(stream, 0, 4, 32)
    m = Model(L, C, NH, V, maxT)
    m.set_params(params)
    loss = m.forward(inp, tgt)
    # logits ~ N(0, C*0.02^2): E[loss] ~ ln V + C*0.02^2/2
    assert abs(loss - (math.log(V) + C * 0.02 ** 2 / 2)) < 0.1
    # zero embeddings: every activation is a bias (all zero), logits are all 0,
    # and the loss is exactly ln V.
    z = params.copy()
    sizes = synth.param_sizes(L, C, V, maxT)
    z[:sizes[0] + sizes[1]] = 0
    m.set_params(z)
    # (exact up to the rounding of log and of the 128-term mean: a few ulps)
    assert abs(m.forward(inp, tgt) - math.log(V)) < 1e-13


def test_causality_and_batch_independence_exact():
    L, C, NH, V, maxT = _cfg("tiny")
    params = synth.init_params(L, C, V, maxT, seed=51)
    inp = synth.zipf_stream(V, 3 * 20, seed=52).reshape(3, 20)
    m = Model(L, C, NH, V, maxT)
    m.set_params(params)
    m.forward(inp)
    base = m.logits().copy()
    t0 = 9
    pert = inp.copy()
    pert[:, t0 + 1:] = (pert[:, t0 + 1:] + 7) % V
    pert[2, :] = (pert[2, :] + 3) % V
    m.forward(pert)
    got = m.logits()
    assert np.array_equal(got[:2, :t0 + 1], base[:2, :t0 + 1])   # future tokens invisible
    assert not np.array_equal(got[:2, t0 + 1:], base[:2, t0 + 1:])
    assert not np.array_equal(got[2], base[2])                   # row 2 changed ...
    pert2 = inp.copy()
    pert2[2, :] = (pert2[2, :] + 3) % V
    m.forward(pert2)
    assert np.array_equal(m.logits()[:2], base[:2])              # ... rows 0,1 untouched


def test_float_variant_tracks_double():
    L, C, NH, V, maxT = _cfg("tiny")
    params = synth.init_params(L, C, V, maxT, seed=61)
    stream = synth.zipf_stream(V, 4 * 32 + 1, seed=62)
    inp, tgt = synth.batch(stream, 0, 4, 32)
    out = {}
    for var in ("f64", "f32"):
        m = Model(L, C, NH, V, maxT, variant=var)
        m.set_params(params)
        loss = m.forward(inp, tgt)
        m.backward()
        m.update(3e-4, 0.9, 0.999, 1e-8, 0.0, 1)
        out[var] = (loss, m.grads().astype(np.float64), m.params().astype(np.float64))
    assert abs(out["f32"][0] - out["f64"][0]) < 1e-5 * out["f64"][0]
    g64, g32 = out["f64"][1], out["f32"][1]
    assert np.linalg.norm(g32 - g64) / np.linalg.norm(g64) < 1e-4


def test_oracle_error_codes():
    m = Model(1, 16, 4, 27, 16)
    with pytest.raises(ValueError):
        m.forward(np.full((2, 4), 27, np.int32))           # id out of range
    with pytest.raises(ValueError):
        m.forward(np.zeros((2, 17), np.int32))             # T > maxT
    m.forward(np.zeros((2, 4), np.int32))
    with pytest.raises(RuntimeError):
        m.backward()                                       # no targets in the last forward
    with pytest.raises(ValueError):
        m.forward(np.zeros((3, 4), np.int32))              # B differs from the first call


# ---------------------------------------------------------------- microGPT variant: RMSNorm
# The page "microGPT 3D" (lesson 04) puts RMSNorm where GPT-2 has LayerNorm.  Read as
# root-mean-square normalisation with eps 1e-5 and a per-channel gain, no shift.

def test_rmsnorm_zero_mean_rows_equal_layernorm():
    """On rows with mean exactly 0 the two normalisations coincide (LayerNorm is pinned
    to the picoGPT worked values above)."""
    rng = np.random.default_rng(71)
    half = rng.normal(size=(16, 24)) * 2.0
    x = np.concatenate([half, -half], axis=1)          # every row sums to exactly 0
    w = rng.normal(size=48)
    ln, _, ln_rstd = ops.layernorm(x, w, np.zeros(48))
    rms, rstd = ops.rmsnorm(x, w)
    assert np.allclose(rms, ln, rtol=1e-13, atol=1e-14)
    assert np.allclose(rstd, ln_rstd, rtol=1e-13)


def test_rmsnorm_moments_and_worked_value():
    rng = np.random.default_rng(72)
    z = rng.normal(size=(32, 97)) * 3 + 1              # non-zero mean: differs from LayerNorm
    o, r = ops.rmsnorm(z, np.ones(97))
    ms = (z * z).mean(-1)
    # unit gain: every output row has mean square ms / (ms + eps), and o / z is one
    # positive constant per row (no shift, no mean subtraction)
    assert np.allclose((o * o).mean(-1), ms / (ms + 1e-5), rtol=1e-12)
    ratio = o / z
    assert np.allclose(ratio, ratio[:, :1], rtol=1e-12) and np.all(ratio > 0)
    ln, _, _ = ops.layernorm(z, np.ones(97), np.zeros(97))
    assert np.max(np.abs(o - ln)) > 0.1
    # by hand: x = (3, 4): mean square 12.5, out = x / sqrt(12.5 + 1e-5)
    o2, _ = ops.rmsnorm(np.array([[3.0, 4.0]]), np.array([1.0, 2.0]))
    assert np.allclose(o2, [[0.848528137423857 * (12.5 / 12.50001) ** 0.5,
                             2 * 1.131370849898476 * (12.5 / 12.50001) ** 0.5]], rtol=1e-14)


def test_rmsnorm_backward_finite_difference():
    rng = np.random.default_rng(73)
    x = rng.normal(size=(3, 10)) + 0.5
    w = rng.normal(size=10)
    dy = rng.normal(size=(3, 10))
    out, rstd = ops.rmsnorm(x, w)
    dx, dw = ops.rmsnorm_backward(dy, x, w, rstd)
    f = lambda: float((ops.rmsnorm(x, w)[0] * dy).sum())
    assert np.allclose(dx, _fd(f, x), atol=1e-8)
    assert np.allclose(dw, _fd(f, w), atol=1e-8)


def test_rmsnorm_model_matches_torch_autograd():
    """The whole microGPT-variant step against torch's rms_norm + autograd (float64)."""
    L, C, NH, V, maxT = _cfg("tiny")
    params = synth.init_params(L, C, V, maxT, seed=74)
    rng = np.random.default_rng(75)
    params = params + rng.normal(scale=0.02, size=params.size).astype(np.float32)
    stream = synth.zipf_stream(V, 4 * 32 + 1, seed=76)
    inp, tgt = synth.batch(stream, 0, 4, 32)
    m = Model(L, C, NH, V, maxT, norm="rmsnorm")
    m.set_params(params)
    loss = m.forward(inp, tgt)
    m.backward()
    tl, tg, tlog = torch_loss_and_grads(params, inp, tgt, L, C, NH, V, maxT, norm="rmsnorm")
    assert abs(loss - tl) <= 1e-12 * abs(tl)
    assert np.allclose(m.logits(), tlog, rtol=1e-10, atol=1e-12)
    g = m.grads()
    sizes = synth.param_sizes(L, C, V, maxT)
    for name, a, b in zip(synth.PARAM_NAMES, np.split(g, np.cumsum(sizes)[:-1]), np.split(tg, np.cumsum(sizes)[:-1])):
        if name in ("ln1b", "ln2b", "lnfb"):
            assert not a.any() and not b.any(), name    # the shifts are carried, unused
            continue
        err = np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)
        assert err < 1e-10, (name, err)
    # and it is a different model from the LayerNorm one on the same weights
    ml = Model(L, C, NH, V, maxT)
    ml.set_params(params)
    assert abs(ml.forward(inp, tgt) - loss) > 1e-6


def test_rmsnorm_model_finite_difference_char_all_params():
    L, C, NH, V, maxT = _cfg("char")
    params = synth.init_params(L, C, V, maxT, seed=77).astype(np.float64)
    params += np.random.default_rng(78).normal(scale=0.05, size=params.size)
    stream = synth.uniform_stream(V, 4 * 16 + 1, seed=79)
    inp, tgt = synth.batch(stream, 0, 4, 16)
    m = Model(L, C, NH, V, maxT, norm="rmsnorm")
    f = _loss_fn(m, params, inp, tgt)
    f()
    m.backward()
    g = m.grads()
    fd = _fd(f, params, h=1e-6)
    assert np.all(np.abs(fd - g) <= 1e-6 * np.abs(g) + 2e-9), np.max(np.abs(fd - g))


# ---------------------------------------------------------------- generation
# picoGPT's "generate" (greedy decode loop; sampling with np.random.choice over the
# last position's distribution, temperature as the article's knob) and llm.c §1.35
# sample_mult.

def test_sample_mult_matches_searchsorted_and_edges():
    rng = np.random.default_rng(81)
    p = rng.random(37)
    p /= p.sum()
    cdf = np.cumsum(p)
    for coin in rng.random(500):
        assert ops.sample_mult(p, coin) == int(np.searchsorted(cdf, coin, side="right"))
    assert ops.sample_mult(np.array([0.0, 0.0, 1.0]), 0.0) == 2     # zero-mass ids are never drawn
    assert ops.sample_mult(np.array([0.25, 0.25, 0.25, 0.25]), 0.5) == 2
    assert ops.sample_mult(np.array([0.3, 0.3, 0.3]), 0.95) == 2    # rounding slack: last id
    # frequencies over a fine grid of coins reproduce the distribution exactly
    coins = (np.arange(100000) + 0.5) / 100000
    counts = np.bincount([ops.sample_mult(p, c) for c in coins[::10]], minlength=37)
    assert np.allclose(counts / counts.sum(), p, atol=2e-4)


def _pico_generate(params, prompt, n_new, cfg, temperature=0.0, coins=None):
    L, C, NH, V, maxT = cfg
    seq = np.array(prompt)
    out = []
    for s in range(n_new):
        logits = picogpt_logits(params, seq, L, C, NH, V, maxT)[:, -1]
        if temperature <= 0:
            nxt = np.argmax(logits, axis=-1)
        else:
            z = logits / temperature
            e = np.exp(z - z.max(-1, keepdims=True))
            p = e / e.sum(-1, keepdims=True)
            nxt = np.array([int(np.searchsorted(np.cumsum(p[b]), coins[b, s], side="right"))
                            for b in range(seq.shape[0])])
        out.append(nxt)
        seq = np.concatenate([seq, nxt[:, None]], axis=1)
    return np.stack(out, axis=1)


def test_generate_greedy_matches_picogpt_loop():
    cfg = _cfg("tiny")
    L, C, NH, V, maxT = cfg
    params = synth.init_params(L, C, V, maxT, seed=82).astype(np.float64)
    params += np.random.default_rng(83).normal(scale=0.05, size=params.size)   # non-flat logits
    prompt = synth.zipf_stream(V, 3 * 5, seed=84).reshape(3, 5)
    m = Model(*cfg)
    m.set_params(params)
    got = m.generate(prompt, 6)
    want = _pico_generate(params, prompt, 6, cfg)
    assert np.array_equal(got, want)
    # each row's continuation depends on that row only
    got1 = m.generate(prompt[1:2], 6)
    assert np.array_equal(got1[0], got[1])


def test_generate_sampling_matches_picogpt_loop_and_low_temperature_is_greedy():
    cfg = _cfg("tiny")
    L, C, NH, V, maxT = cfg
    params = synth.init_params(L, C, V, maxT, seed=85).astype(np.float64)
    params += np.random.default_rng(86).normal(scale=0.05, size=params.size)
    prompt = synth.zipf_stream(V, 2 * 4, seed=87).reshape(2, 4)
    coins = np.random.default_rng(88).random((2, 5))
    m = Model(*cfg)
    m.set_params(params)
    for tau in (1.0, 0.7):
        got = m.generate(prompt, 5, temperature=tau, coins=coins)
        want = _pico_generate(params, prompt, 5, cfg, temperature=tau, coins=coins)
        assert np.array_equal(got, want), tau
    # as the temperature goes to 0 the distribution collapses onto the argmax
    cold = m.generate(prompt, 5, temperature=1e-4, coins=coins)
    assert np.array_equal(cold, m.generate(prompt, 5))


def test_rmsnorm_model_forward_matches_numpy_statement():
    """The RMSNorm model's logits against a numpy restatement of the same forward."""
    L, C, NH, V, maxT = _cfg("tiny")
    params = synth.init_params(L, C, V, maxT, seed=89).astype(np.float64)
    params += np.random.default_rng(90).normal(scale=0.05, size=params.size)
    inp = synth.zipf_stream(V, 2 * 12, seed=91).reshape(2, 12)
    m = Model(L, C, NH, V, maxT, norm="rmsnorm")
    m.set_params(params)
    m.forward(inp)
    want = picogpt_logits(params, inp, L, C, NH, V, maxT, norm="rmsnorm")
    assert np.allclose(m.logits(), want, rtol=1e-11, atol=1e-12)
    assert not np.allclose(want, picogpt_logits(params, inp, L, C, NH, V, maxT), atol=1e-3)
