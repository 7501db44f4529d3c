"""The sampling loop (crop to the block size, last-position logits,
temperature, top-k, multinomial draw; no KV cache), run on the oracle's model
on CPU. The library plugs its own forward into the same loop; the padding
scheme it uses (context padded to the model's T, logits read at position t-1)
is checked here on the oracle: causality makes it give the same tokens as
running each context at its exact length."""
import numpy as np

from decoder_only_transformer_06_b300.generate import generate, sample_next
from oracle import CONFIGS
from oracle import gpt2_oracle as O


def test_top1_is_argmax_and_masked_tokens_are_never_drawn():
    rng = np.random.default_rng(0)
    z = rng.normal(size=(6, 50))
    got = sample_next(z, 0.8, 1, np.random.default_rng(1))
    assert np.array_equal(got, z.argmax(axis=1))
    draws = np.concatenate([sample_next(z, 1.3, 5, np.random.default_rng(s)) for s in range(300)])
    top5 = np.argsort(z, axis=1)[:, -5:]
    rows = np.tile(np.arange(6), 300)
    assert all(d in top5[r] for d, r in zip(draws, rows))


def test_draw_frequencies_follow_the_tempered_softmax():
    z = np.array([[2.0, 1.0, 0.5, -1.0, 0.0]])
    T = 0.7
    p = np.exp(z[0] / T) / np.exp(z[0] / T).sum()
    rng = np.random.default_rng(7)
    n = 200000
    counts = np.bincount(sample_next(np.repeat(z, n, axis=0), T, None, rng), minlength=5)
    # 5 binomial standard deviations
    assert np.all(np.abs(counts / n - p) <= 5 * np.sqrt(p * (1 - p) / n))


def test_padded_context_gives_the_exact_length_tokens_and_the_crop_applies():
    c = CONFIGS["tiny"]                       # block_size 64
    params = O.init_params(c, 5)

    def exact(ctx):
        _, logits, _ = O.forward(params, c, ctx)
        return logits[:, -1, :]

    def padded(ctx):
        b, t = ctx.shape
        buf = np.zeros((b, c.block_size), dtype=np.int64)
        buf[:, :t] = ctx
        _, logits, _ = O.forward(params, c, buf)
        return logits[:, t - 1, :]

    prompt = np.random.default_rng(3).integers(0, c.vocab_size, size=(2, 5))
    n_new = c.block_size + 6                  # the context outgrows the block: cropped
    a = generate(exact, prompt, n_new, c.block_size, temperature=0.8, top_k=20, seed=11)
    b = generate(padded, prompt, n_new, c.block_size, temperature=0.8, top_k=20, seed=11)
    assert a.shape == (2, 5 + n_new)
    assert np.array_equal(a[:, :5], prompt)
    assert np.array_equal(a, b)
    assert a.min() >= 0 and a.max() < c.vocab_size
