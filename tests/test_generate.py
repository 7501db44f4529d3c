"""Generation on the CPU side: the oracle's sampler against what the pages fix
and the mathematics implies, and the generation loop's context handling
(padding to the model's T, crop to the block size) on the oracle's model.
The library runs the same loop on the GPU (tests/test_gpu_generate.py)."""
import numpy as np

import synthdata
from decoder_only_transformer_06_b300.generate import draw_uniforms
from oracle import CONFIGS
from oracle import gpt2_oracle as O


def _u(n, seed=0):
    return synthdata.uniforms(seed, np.arange(n))


def test_top1_is_argmax_and_masked_tokens_are_never_drawn():
    rng = np.random.default_rng(0)
    z = rng.normal(size=(6, 50))
    assert np.array_equal(O.sample_tokens(z, 0.8, 1, _u(6)), z.argmax(axis=1))
    assert np.array_equal(O.sample_tokens(z, 0.0, None, _u(6)), z.argmax(axis=1))
    draws = np.concatenate([O.sample_tokens(z, 1.3, 5, _u(6, s)) for s in range(300)])
    top5 = np.argsort(z, axis=1)[:, -5:]
    rows = np.tile(np.arange(6), 300)
    assert all(d in top5[r] for d, r in zip(draws, rows))


def test_draw_frequencies_follow_the_tempered_softmax():
    z = np.array([[2.0, 1.0, 0.5, -1.0, 0.0]])
    T = 0.7
    p = np.exp(z[0] / T) / np.exp(z[0] / T).sum()
    n = 200000
    counts = np.bincount(O.sample_tokens(np.repeat(z, n, axis=0), T, None, _u(n, 7)), minlength=5)
    # 5 binomial standard deviations
    assert np.all(np.abs(counts / n - p) <= 5 * np.sqrt(p * (1 - p) / n))


def test_inverse_cdf_closed_form_on_equal_logits():
    """Equal logits: p uniform over the V entries, so the token is floor(u V)
    (u kept away from the cell boundaries)."""
    V = 97
    u = (np.arange(40) + 0.5) / 40
    got = O.sample_tokens(np.zeros((40, V)), 1.0, None, u)
    assert np.array_equal(got, np.floor(u * V).astype(np.int64))


def test_top_k_keeps_ties_with_the_kth_value():
    """The pages' mask sets logits < the k-th largest to -inf: entries equal to
    it stay. z = [3, 2, 2, 1], k = 2 keeps {0, 1, 2} with weights e^3, e^2, e^2."""
    z = np.array([[3.0, 2.0, 2.0, 1.0]])
    w = np.exp(np.array([3.0, 2.0, 2.0]))
    c = np.cumsum(w) / w.sum()
    for u, want in ((0.5 * c[0], 0), (0.5 * (c[0] + c[1]), 1), (0.5 * (c[1] + 1.0), 2)):
        assert O.sample_tokens(z, 1.0, 2, np.array([u]))[0] == want


def test_uniform_draws_are_the_documented_splitmix64_stream():
    """The generation loop's uniforms: top 24 bits of SplitMix64 output
    step*B + row, times 2^-24 (fp32-exact)."""
    B = 5
    for step in (0, 3):
        got = draw_uniforms(1234, step, B)
        raw = synthdata.splitmix64(1234, np.arange(step * B, step * B + B))
        want = (raw >> np.uint64(40)).astype(np.float64) * 2.0 ** -24
        assert got.dtype == np.float32 and np.array_equal(got.astype(np.float64), want)


def oracle_generate(params, cfg, prompt, n_new, temperature, top_k, uniforms, pad_to=None):
    """The pages' loop on the oracle: crop the context to the block size, the
    last position's logits (padded to pad_to with token 0 when given), sample."""
    idx = np.asarray(prompt, dtype=np.int64)
    for s in range(n_new):
        ctx = idx[:, -cfg.block_size:]
        if pad_to:
            b, t = ctx.shape
            buf = np.zeros((b, pad_to), dtype=np.int64)
            buf[:, :t] = ctx
            _, logits, _ = O.forward(params, cfg, buf)
            last = logits[:, t - 1, :]
        else:
            _, logits, _ = O.forward(params, cfg, ctx)
            last = logits[:, -1, :]
        nxt = O.sample_tokens(last, temperature, top_k, uniforms[s, :idx.shape[0]])
        idx = np.concatenate([idx, nxt[:, None]], axis=1)
    return idx


def test_padded_context_gives_the_exact_length_tokens_and_the_crop_applies():
    c = CONFIGS["tiny"]                       # block_size 64
    params = O.init_params(c, 5)
    prompt = np.random.default_rng(3).integers(0, c.vocab_size, size=(2, 5))
    n_new = c.block_size + 6                  # the context outgrows the block: cropped
    u = np.stack([draw_uniforms(11, s, 2) for s in range(n_new)])
    a = oracle_generate(params, c, prompt, n_new, 0.8, 20, u)
    b = oracle_generate(params, c, prompt, n_new, 0.8, 20, u, pad_to=c.block_size)
    assert a.shape == (2, 5 + n_new)
    assert np.array_equal(a[:, :5], prompt)
    assert np.array_equal(a, b)
    assert a.min() >= 0 and a.max() < c.vocab_size
