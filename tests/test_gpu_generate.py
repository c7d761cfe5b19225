"""GPU parity of autoregressive generation (picoGPT's generate loop with a key/value
cache; llm.c section 1.35 sample_mult) against the CPU oracle's full-recompute loop.

Where floating point decides an id (argmax, the coin's place in the cumulative
distribution), exact agreement is required in fp32 mode; in bf16 mode each chosen id
must be a valid choice under the oracle's distribution given the GPU's own history
(a near-maximal logit; a cumulative interval that contains the coin up to the bf16
logits' error)."""
import numpy as np
import pytest

from gpt_train_step_arena_b300 import synth
from oracle.oracle import Model as Oracle

from .gpu_util import cfg_shape, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def G():
    from gpt_train_step_arena_b300.model import GPT2
    return GPT2


def _params(cfg, seed, noise):
    L, C, NH, V, maxT = cfg
    p = synth.init_params(L, C, V, maxT, seed=seed)
    if noise:
        p = p + np.random.default_rng(seed + 1).normal(scale=noise, size=p.size).astype(np.float32)
    return p


def _oracle_last_logits(cfg, params, seq, norm="layernorm"):
    o = Oracle(*cfg, norm=norm)
    o.set_params(params)
    o.forward(seq)
    return o.logits()[:, -1]


def _check_valid(cfg, params, prompt, got, temperature, coins, logit_tol, cdf_tol, norm="layernorm"):
    """Every id the GPU chose is a valid choice under the oracle's distribution after the
    GPU's own history."""
    B, n_new = got.shape
    seq = np.array(prompt)
    for s in range(n_new):
        ref = _oracle_last_logits(cfg, params, seq, norm)
        for b in range(B):
            i = got[b, s]
            assert 0 <= i < cfg[3]
            if temperature <= 0:
                assert ref[b, i] >= ref[b].max() - logit_tol, (s, b, ref[b, i], ref[b].max())
            else:
                z = ref[b] / temperature
                p = np.exp(z - z.max())
                p /= p.sum()
                cdf = np.cumsum(p)
                lo = cdf[i - 1] if i > 0 else 0.0
                c = coins[b, s]
                assert lo - cdf_tol <= c < cdf[i] + cdf_tol, (s, b, lo, c, cdf[i])
        seq = np.concatenate([seq, got[:, s:s + 1]], axis=1)


@pytest.mark.parametrize("norm", ["layernorm", "rmsnorm"])
def test_greedy_fp32_tiny_equals_oracle(G, norm):
    cfg = cfg_shape("tiny")
    L, C, NH, V, maxT = cfg
    params = _params(cfg, 90, 0.05)
    prompt = synth.zipf_stream(V, 3 * 5, seed=91).reshape(3, 5)
    g = G(*cfg, precision="fp32", norm=norm)
    g.set_params(params)
    got = g.generate(prompt, 7)
    o = Oracle(*cfg, norm=norm)
    o.set_params(params)
    want = o.generate(prompt, 7)
    assert np.array_equal(got, want)
    # the cached decode reproduces the full forward: last step's logits vs the oracle
    seq = np.concatenate([prompt, got[:, :-1]], axis=1)
    ref = _oracle_last_logits(cfg, params, seq, norm)
    last = g.gen_logits(3)
    assert rel_l2(last, ref) <= 1e-4
    assert np.max(np.abs(last - ref)) <= 1e-4 * np.max(np.abs(ref))
    g.close()


@pytest.mark.parametrize("tau", [1.0, 0.7])
def test_sampling_fp32_tiny_equals_oracle(G, tau):
    cfg = cfg_shape("tiny")
    L, C, NH, V, maxT = cfg
    params = _params(cfg, 92, 0.05)
    prompt = synth.zipf_stream(V, 2 * 6, seed=93).reshape(2, 6)
    coins = np.random.default_rng(94).random((2, 9)).astype(np.float32)
    g = G(*cfg, precision="fp32")
    g.set_params(params)
    got = g.generate(prompt, 9, temperature=tau, coins=coins)
    o = Oracle(*cfg)
    o.set_params(params)
    want = o.generate(prompt, 9, temperature=tau, coins=coins.astype(np.float64))
    if not np.array_equal(got, want):
        # only a coin within rounding of a cumulative boundary may split the two
        _check_valid(cfg, params, prompt, got, tau, coins, 0.0, 1e-5)
    g.close()


def test_greedy_and_sampling_bf16_gpt2_124m_shapes(G):
    """124M shapes (L=12, C=768, V=50257) on the tensor-core path: every choice valid."""
    cfg = cfg_shape("gpt2_124m_small")
    L, C, NH, V, maxT = cfg
    params = _params(cfg, 95, 0.0)
    prompt = synth.zipf_stream(V, 4 * 16, seed=96).reshape(4, 16)
    g = G(*cfg, precision="bf16")
    g.set_params(params)
    greedy = g.generate(prompt, 6)
    ref = _oracle_last_logits(cfg, params, np.concatenate([prompt, greedy[:, :-1]], axis=1))
    assert rel_l2(g.gen_logits(4), ref) <= 3e-2
    _check_valid(cfg, params, prompt, greedy, 0.0, None, 0.05 * np.abs(ref).max(), 0.0)
    coins = np.random.default_rng(97).random((4, 6)).astype(np.float32)
    sampled = g.generate(prompt, 6, temperature=1.0, coins=coins)
    _check_valid(cfg, params, prompt, sampled, 1.0, coins, 0.0, 2e-3)
    g.close()


def test_cache_decode_matches_own_full_forward_bf16(G):
    """The cached decode of a long continuation against the training forward of the same
    library over the whole sequence (different attention kernels, same model)."""
    cfg = cfg_shape("gpt2_124m_small")
    L, C, NH, V, maxT = cfg
    params = _params(cfg, 98, 0.0)
    prompt = synth.zipf_stream(V, 2 * 40, seed=99).reshape(2, 40)
    g = G(*cfg, precision="bf16")
    g.set_params(params)
    got = g.generate(prompt, 24)
    last = g.gen_logits(2)
    seq = np.concatenate([prompt, got[:, :-1]], axis=1)
    g.forward(seq)
    full = g.logits(2, seq.shape[1])[:, -1]
    assert rel_l2(last, full) <= 2e-2
    g.close()


def test_edges_and_errors(G):
    from gpt_train_step_arena_b300 import _native as N
    from gpt_train_step_arena_b300.model import GPT2Error
    cfg = cfg_shape("tiny")
    L, C, NH, V, maxT = cfg
    params = _params(cfg, 100, 0.05)
    g = G(*cfg, precision="fp32")
    g.set_params(params)
    prompt = synth.zipf_stream(V, 2 * 4, seed=101).reshape(2, 4)
    assert g.generate(prompt, 0).shape == (2, 0)
    with pytest.raises(GPT2Error) as e:
        g.generate(prompt, maxT - 4 + 2)                    # T0 + n_new - 1 > maxT
    assert e.value.code == N.GPT2_ERR_SHAPE
    bad = prompt.copy()
    bad[1, 2] = V
    with pytest.raises(GPT2Error) as e:
        g.generate(bad, 2)
    assert e.value.code == N.GPT2_ERR_TOKEN
    with pytest.raises(GPT2Error) as e:
        g.generate(prompt, 2, temperature=1.0)              # sampling without coins
    assert e.value.code == N.GPT2_ERR_ARG
    with pytest.raises(GPT2Error) as e:
        g.generate(prompt, 2, temperature=1.0, coins=np.full((2, 2), 1.0, np.float32))
    assert e.value.code == N.GPT2_ERR_ARG
    # the longest continuation: the last forward covers all maxT positions
    full = synth.zipf_stream(V, 1 * (maxT - 3), seed=102).reshape(1, maxT - 3)
    got = g.generate(full, 4)
    o = Oracle(*cfg)
    o.set_params(params)
    assert np.array_equal(got, o.generate(full, 4))
    # a one-token prompt, then another batch size (the cache is rebuilt)
    one = prompt[:, :1]
    assert np.array_equal(g.generate(one, 5), o.generate(one, 5))
    three = synth.zipf_stream(V, 3 * 3, seed=103).reshape(3, 3)
    assert np.array_equal(g.generate(three, 3), o.generate(three, 3))
    # run to run: bitwise the same ids and logits
    a = g.generate(three, 3)
    la = g.gen_logits(3)
    b = g.generate(three, 3)
    assert np.array_equal(a, b) and np.array_equal(la, g.gen_logits(3))
    g.close()
