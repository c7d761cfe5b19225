"""GPU parity: the CUDA library (through the C ABI) against the CPU oracle on the same
seeded inputs, for both precision modes, plus the invariances and error paths of the
training step.  All tests need a B300 (marker gpu)."""
import math

import numpy as np
import pytest

from gpt_train_step_arena_b300 import synth
from oracle.oracle import Model as Oracle

from .gpu_util import TOL, assert_grads_close, cfg_shape, per_tensor_errors, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def G():
    from gpt_train_step_arena_b300.model import GPT2
    return GPT2


def _run_one_step(G, name, precision, B=None, T=None, seed=42, variant="f64", norm="layernorm"):
    c = synth.WORKLOADS[name]
    L, C, NH, V, maxT = cfg_shape(name)
    B = B or c["B"]
    T = T or c["T"]
    params = synth.init_params(L, C, V, maxT, seed=seed)
    stream = synth.token_stream(c, steps=1)
    if stream.size < B * T + 1:
        stream = synth.token_stream(c, steps=(B * T) // (c["B"] * c["T"]) + 2)
    inp, tgt = synth.batch(stream, 0, B, T)
    hp = (c["lr"], c["b1"], c["b2"], c["eps"], c["wd"])

    o = Oracle(L, C, NH, V, maxT, variant=variant, norm=norm)
    o.set_params(params)
    o.forward(inp)
    ref_logits = o.logits().copy()
    ref_loss = o.forward(inp, tgt)
    ref_losses = o.losses().copy()
    o.backward()
    ref_grads = o.grads().copy()
    o.update(*hp, 1)
    ref_params = o.params().copy()

    # a fresh handle per pass so the logits of a forward without targets are kept
    g = G(L, C, NH, V, maxT, precision=precision, norm=norm)
    g.set_params(params)
    assert g.forward(inp) == -1.0
    logits = g.logits(B, T)
    g.close()
    g = G(L, C, NH, V, maxT, precision=precision, norm=norm)
    g.set_params(params)
    loss = g.forward(inp, tgt)
    tok_back, tgt_back = g.ids(B, T)
    losses = g.losses(B, T)
    g.backward()
    grads = g.grads()
    g.update(*hp, 1)
    new_params = g.params()
    g.close()
    return dict(inp=inp, tgt=tgt, tok_back=tok_back, tgt_back=tgt_back, loss=loss, ref_loss=ref_loss,
                losses=losses, ref_losses=ref_losses, logits=logits, ref_logits=ref_logits,
                grads=grads, ref_grads=ref_grads, params=new_params, ref_params=ref_params,
                init=params, shape=(L, C, V, maxT))


@pytest.mark.parametrize("precision", ["fp32", "bf16"])
def test_tiny_one_step(G, precision):
    r = _run_one_step(G, "tiny", precision)
    tol = TOL[precision]
    L, C, V, maxT = r["shape"]
    assert np.array_equal(r["tok_back"], r["inp"]) and np.array_equal(r["tgt_back"], r["tgt"])
    assert abs(r["loss"] - r["ref_loss"]) <= tol["loss"] * abs(r["ref_loss"]), (r["loss"], r["ref_loss"])
    if tol["logits"]:
        assert rel_l2(r["logits"], r["ref_logits"]) <= tol["logits"]
        assert np.max(np.abs(r["logits"] - r["ref_logits"])) <= tol["logits"] * np.max(np.abs(r["ref_logits"]))
    assert_grads_close(r["grads"], r["ref_grads"], L, C, V, maxT, tol["grads"])
    # AdamW (fp32 master in both modes, so its arithmetic is checked in fp32 mode): at
    # t=1 the step is lr*g/(|g|+eps), so compare it where the reference gradient is
    # well above the gradient error; elsewhere the step's sign is set by noise.
    if precision == "fp32":
        g = r["ref_grads"]
        d_got = r["params"].astype(np.float64) - r["init"]
        d_ref = r["ref_params"] - r["init"]
        lr = synth.WORKLOADS["tiny"]["lr"]
        well = np.abs(g) > 1e-3 * np.sqrt(np.mean(g * g))
        assert np.max(np.abs(d_got - d_ref)[well]) <= 1e-3 * lr
        # |step| <= lr at t=1 with wd = 0, up to the fp32 rounding of the new parameter
        slack = np.spacing(np.abs(r["init"]).astype(np.float32)).astype(np.float64)
        assert np.all(np.abs(d_got) <= lr * (1 + 1e-6) + slack)


def test_tiny_bf16_logits_close(G):
    r = _run_one_step(G, "tiny", "bf16")
    # bf16 logits: relative-L2 within a few bf16 ulps of the activations
    assert rel_l2(r["logits"], r["ref_logits"]) <= 3e-2


def test_char_fp32_fifty_steps_vs_float_oracle(G):
    """Loss curve of 50 AdamW steps against the float oracle (the listing's precision)."""
    c = synth.WORKLOADS["char"]
    L, C, NH, V, maxT = cfg_shape("char")
    B, T, steps = c["B"], c["T"], c["steps"]
    params = synth.init_params(L, C, V, maxT, seed=42)
    stream = synth.token_stream(c, steps=steps)
    hp = (c["lr"], c["b1"], c["b2"], c["eps"], c["wd"])
    o = Oracle(L, C, NH, V, maxT, variant="f32")
    o.set_params(params)
    g = G(L, C, NH, V, maxT, precision="fp32")
    g.set_params(params)
    for s in range(steps):
        inp, tgt = synth.batch(stream, s, B, T)
        lr_ = o.forward(inp, tgt)
        o.backward()
        o.update(*hp, s + 1)
        lg = g.forward(inp, tgt)
        g.backward()
        g.update(*hp, s + 1)
        rel = abs(lg - lr_) / abs(lr_)
        assert rel <= (1e-5 if s < 10 else 1e-3), (s, lg, lr_)
    g.close()


def test_gpt2_124m_small_fp32(G):
    """GPT-2 124M shapes at B=4, T=64 in strict fp32 against the double oracle."""
    r = _run_one_step(G, "gpt2_124m_small", "fp32")
    L, C, V, maxT = r["shape"]
    assert abs(r["loss"] - r["ref_loss"]) <= 1e-5 * r["ref_loss"]
    assert rel_l2(r["logits"], r["ref_logits"]) <= 1e-4
    assert_grads_close(r["grads"], r["ref_grads"], L, C, V, maxT, 1e-3)


def test_gpt2_124m_small_bf16(G):
    r = _run_one_step(G, "gpt2_124m_small", "bf16")
    L, C, V, maxT = r["shape"]
    assert abs(r["loss"] - r["ref_loss"]) <= 1e-2 * r["ref_loss"]
    assert_grads_close(r["grads"], r["ref_grads"], L, C, V, maxT, 3e-2)


@pytest.mark.parametrize("B,T", [(1, 1), (3, 17), (2, 32)])
def test_ragged_shapes_fp32(G, B, T):
    """Empty-ish and ragged batches (T not a multiple of any tile, B=1, T=1)."""
    L, C, NH, V, maxT = cfg_shape("tiny")
    params = synth.init_params(L, C, V, maxT, seed=7)
    stream = synth.zipf_stream(V, B * T + 1, seed=8)
    inp, tgt = synth.batch(stream, 0, B, T)
    o = Oracle(L, C, NH, V, maxT)
    o.set_params(params)
    ref = o.forward(inp, tgt)
    o.backward()
    g = G(L, C, NH, V, maxT, precision="fp32")
    g.set_params(params)
    loss = g.forward(inp, tgt)
    g.backward()
    assert abs(loss - ref) <= 1e-5 * ref
    assert_grads_close(g.grads(), o.grads(), L, C, V, maxT, 1e-3)
    g.close()


def test_odd_vocab_char_one_step(G):
    """V=27 is padded to 128 on the device; padded rows stay zero through AdamW."""
    r = _run_one_step(G, "char", "fp32")
    L, C, V, maxT = r["shape"]
    assert abs(r["loss"] - r["ref_loss"]) <= 1e-5 * r["ref_loss"]
    assert_grads_close(r["grads"], r["ref_grads"], L, C, V, maxT, 1e-3)


@pytest.mark.parametrize("precision", ["fp32", "bf16"])
def test_causality_and_batch_independence(G, precision):
    L, C, NH, V, maxT = cfg_shape("tiny")
    params = synth.init_params(L, C, V, maxT, seed=51)
    inp = synth.zipf_stream(V, 3 * 20, seed=52).reshape(3, 20)
    g = G(L, C, NH, V, maxT, precision=precision)
    g.set_params(params)
    g.forward(inp)
    base = g.logits(3, 20)
    t0 = 9
    pert = inp.copy()
    pert[:, t0 + 1:] = (pert[:, t0 + 1:] + 7) % V
    g.forward(pert)
    got = g.logits(3, 20)
    assert np.array_equal(got[:, :t0 + 1], base[:, :t0 + 1])
    pert2 = inp.copy()
    pert2[2, :] = (pert2[2, :] + 3) % V
    g.forward(pert2)
    assert np.array_equal(g.logits(3, 20)[:2], base[:2])
    g.close()


@pytest.mark.parametrize("precision", ["fp32", "bf16"])
def test_run_to_run_bitwise_determinism(G, precision):
    L, C, NH, V, maxT = cfg_shape("tiny")
    params = synth.init_params(L, C, V, maxT, seed=5)
    stream = synth.zipf_stream(V, 4 * 32 + 1, seed=6)
    inp, tgt = synth.batch(stream, 0, 4, 32)
    outs = []
    for _ in range(2):
        g = G(L, C, NH, V, maxT, precision=precision)
        g.set_params(params)
        loss = g.forward(inp, tgt)
        g.backward()
        g.update(3e-4, 0.9, 0.999, 1e-8, 0.1, 1)
        outs.append((loss, g.grads(), g.params()))
        g.close()
    assert outs[0][0] == outs[1][0]
    assert np.array_equal(outs[0][1], outs[1][1])
    assert np.array_equal(outs[0][2], outs[1][2])


def test_error_paths_never_fault(G):
    from gpt_train_step_arena_b300.model import GPT2Error
    from gpt_train_step_arena_b300 import _native as N
    L, C, NH, V, maxT = cfg_shape("tiny")
    g = G(L, C, NH, V, maxT, precision="fp32")
    g.set_params(synth.init_params(L, C, V, maxT))
    with pytest.raises(GPT2Error) as e:
        g.backward()                                       # no forward yet
    assert e.value.code == N.GPT2_ERR_STATE
    bad = np.zeros((2, 8), np.int32)
    bad[1, 3] = V                                          # id out of range
    with pytest.raises(GPT2Error) as e:
        g.forward(bad, np.zeros((2, 8), np.int32))
    assert e.value.code == N.GPT2_ERR_TOKEN
    with pytest.raises(GPT2Error) as e:
        g.backward()                                       # failed forward cannot feed it
    assert e.value.code == N.GPT2_ERR_STATE
    tg = np.zeros((2, 8), np.int32)
    tg[0, 0] = -1                                          # target out of range
    with pytest.raises(GPT2Error) as e:
        g.forward(np.zeros((2, 8), np.int32), tg)
    assert e.value.code == N.GPT2_ERR_TOKEN
    with pytest.raises(GPT2Error) as e:
        g.forward(np.zeros((3, 8), np.int32))              # B differs from the first call
    assert e.value.code == N.GPT2_ERR_SHAPE
    with pytest.raises(GPT2Error) as e:
        g.update(1e-3, 0.9, 0.999, 1e-8, 0.0, 0)           # t must be >= 1
    assert e.value.code == N.GPT2_ERR_ARG
    # the handle is still usable after all of the above
    loss = g.forward(np.zeros((2, 8), np.int32), np.zeros((2, 8), np.int32))
    assert math.isfinite(loss)
    g.backward()
    g.update(1e-3, 0.9, 0.999, 1e-8, 0.0, 1)
    g.close()
    with pytest.raises(GPT2Error) as e:
        G(L, C, 5, V, maxT)                                # C % H != 0
    assert e.value.code == N.GPT2_ERR_ARG
    g = G(L, C, NH, V, 8, precision="fp32")
    with pytest.raises(GPT2Error) as e:
        g.forward(np.zeros((1, 9), np.int32))              # T > maxT
    assert e.value.code == N.GPT2_ERR_SHAPE
    g.close()


# ---------------------------------------------------------------- microGPT variant (RMSNorm)
@pytest.mark.parametrize("precision", ["fp32", "bf16"])
def test_rmsnorm_variant_tiny_one_step(G, precision):
    r = _run_one_step(G, "tiny", precision, norm="rmsnorm")
    tol = TOL[precision]
    L, C, V, maxT = r["shape"]
    assert abs(r["loss"] - r["ref_loss"]) <= tol["loss"] * abs(r["ref_loss"]), (r["loss"], r["ref_loss"])
    if tol["logits"]:
        assert rel_l2(r["logits"], r["ref_logits"]) <= tol["logits"]
    assert_grads_close(r["grads"], r["ref_grads"], L, C, V, maxT, tol["grads"])
    # the shift tensors are unused: their gradients are exactly zero on the device too
    sizes = synth.param_sizes(L, C, V, maxT)
    for name, gpart in zip(synth.PARAM_NAMES, np.split(r["grads"], np.cumsum(sizes)[:-1])):
        if name in ("ln1b", "ln2b", "lnfb"):
            assert not gpart.any(), name


@pytest.mark.parametrize("precision", ["fp32", "bf16"])
def test_rmsnorm_variant_gpt2_124m_small(G, precision):
    """124M shapes at B=4, T=64 with RMSNorm, against the double oracle's RMSNorm model."""
    r = _run_one_step(G, "gpt2_124m_small", precision, norm="rmsnorm")
    L, C, V, maxT = r["shape"]
    tol = TOL[precision]
    assert abs(r["loss"] - r["ref_loss"]) <= tol["loss"] * r["ref_loss"]
    if tol["logits"]:
        assert rel_l2(r["logits"], r["ref_logits"]) <= tol["logits"]
    assert_grads_close(r["grads"], r["ref_grads"], L, C, V, maxT, tol["grads"])



def test_bounded_wait_expiry_reports_timeout_and_handle_stays_usable(G):
    """A device wait that nothing completes gives up after its limit, raises the timeout
    flag, and the host reports GPT2_ERR_TIMEOUT; the handle then trains on exactly as a
    fresh one does."""
    import time
    from gpt_train_step_arena_b300 import _native as N
    L, C, NH, V, maxT = cfg_shape("tiny")
    params = synth.init_params(L, C, V, maxT, seed=3)
    inp, tgt = synth.batch(synth.zipf_stream(V, 2 * 16 + 1, seed=4), 0, 2, 16)
    g = G(L, C, NH, V, maxT, precision="bf16")
    assert N.lib.gpt2_check_bounded_wait(g.h, 1000) == N.GPT2_ERR_STATE     # no forward yet
    g.set_params(params)
    g.forward(inp, tgt)
    t0 = time.perf_counter()
    rc = N.lib.gpt2_check_bounded_wait(g.h, 20000)                           # 20 ms limit
    elapsed = time.perf_counter() - t0
    assert rc == N.GPT2_ERR_TIMEOUT, rc
    assert b"timeout" in N.lib.gpt2_last_error(g.h)
    assert 0.015 <= elapsed < 5.0, elapsed                                   # it waited, then gave up
    # still usable: one step equals the same step on a fresh handle
    g.set_params(params)
    loss = g.forward(inp, tgt)
    g.backward()
    grads = g.grads()
    g.close()
    f = G(L, C, NH, V, maxT, precision="bf16")
    f.set_params(params)
    assert f.forward(inp, tgt) == loss
    f.backward()
    assert np.array_equal(f.grads(), grads)
    f.close()


@pytest.mark.parametrize("precision", ["bf16", "tf32"])
def test_split_k_weight_gradients_whole_step(G, precision):
    """1,024 tokens per step on the tiny model: every weight-gradient product is split over
    K (4 splits of 256 tokens each) and summed in the kernel by the last split to finish, on
    one shared workspace holding products of different sizes, twice in a row."""
    L, C, NH, V, maxT = cfg_shape("tiny")
    params = synth.init_params(L, C, V, maxT, seed=21)
    stream = synth.zipf_stream(V, 2 * 32 * 32 + 1, seed=22)
    o = Oracle(L, C, NH, V, maxT)
    g = G(L, C, NH, V, maxT, precision=precision)
    g.set_params(params)
    o.set_params(params)
    for step in range(2):
        inp, tgt = synth.batch(stream, step, 32, 32)
        ref = o.forward(inp, tgt)
        o.backward()
        loss = g.forward(inp, tgt)
        g.backward()
        assert abs(loss - ref) <= 1e-2 * ref
        assert_grads_close(g.grads(), o.grads(), L, C, V, maxT, 3e-2)
        o.release_acts()
    g.close()
