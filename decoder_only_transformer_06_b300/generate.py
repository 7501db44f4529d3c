"""Sampling from a trained model, as the pages' generate loop does it ("Let's
reproduce GPT-2", the sampling loop; nanoGPT guide, sample.py): crop the
context to the block size, take the logits of the last position, divide by the
temperature, keep the top k, softmax, draw one token, append, repeat. There is
no KV cache: every new token runs the forward again on the whole context.

The loop takes a `last_logits(ctx)` callable (ctx: int [B', t] -> float
[B', V], the logits of position t-1 of each row), so that one loop serves the
library (`library_last_logits`) and any other model of the same method.
Randomness: one numpy Generator seeded by the caller, one uniform draw per row
per token.
"""
import numpy as np


def sample_next(logits, temperature, top_k, rng):
    """One token per row from logits [B, V]: z = logits / temperature; with
    top_k, entries below the k-th largest of the row become -inf; p =
    softmax(z); the token is the first index whose cumulative p exceeds a
    uniform draw (the pages' topk mask keeps ties with the k-th value too)."""
    if temperature <= 0:
        raise ValueError("temperature must be > 0")
    z = np.asarray(logits, dtype=np.float64) / temperature
    if z.ndim != 2:
        raise ValueError("logits must be [B, V]")
    V = z.shape[1]
    if top_k is not None and 0 < top_k < V:
        kth = np.partition(z, V - top_k, axis=1)[:, V - top_k][:, None]
        z = np.where(z < kth, -np.inf, z)
    z = z - z.max(axis=1, keepdims=True)
    p = np.exp(z)
    p /= p.sum(axis=1, keepdims=True)
    cdf = np.cumsum(p, axis=1)
    u = rng.random(z.shape[0])
    j = (cdf <= u[:, None]).sum(axis=1)
    # a draw above the rounded total falls to the last token that can be drawn
    last = V - 1 - np.argmax(p[:, ::-1] > 0, axis=1)
    return np.where(j >= V, last, j).astype(np.int64)


def generate(last_logits, prompt, max_new_tokens, block_size, temperature=1.0, top_k=None, seed=0):
    """Extend every row of `prompt` (int [B, t0], t0 >= 1) by max_new_tokens
    sampled tokens; returns int64 [B, t0 + max_new_tokens]."""
    idx = np.asarray(prompt, dtype=np.int64)
    if idx.ndim != 2 or idx.shape[1] < 1:
        raise ValueError("prompt must be [B, t0] with t0 >= 1")
    rng = np.random.default_rng(seed)
    for _ in range(max_new_tokens):
        ctx = idx[:, -block_size:]
        nxt = sample_next(last_logits(ctx), temperature, top_k, rng)
        idx = np.concatenate([idx, nxt[:, None]], axis=1)
    return idx


def library_last_logits(model):
    """`last_logits` for a gpt2.GPT2 model of batch B and sequence length T.
    The context (B' <= B rows of t <= T tokens) is padded with token 0 to
    [B, T]: causal attention makes the logits of position t-1 independent of
    the padding. One forward (without targets) per call; the logits of the
    rows' positions t-1 are copied back. Use block_size = T with it."""
    import torch

    B, T = model.cfg.batch_size, model.cfg.seq_len

    def last_logits(ctx):
        ctx = np.asarray(ctx)
        b, t = ctx.shape
        if b > B or t > T or t < 1:
            raise ValueError(f"context {ctx.shape} does not fit the model's [{B}, {T}]")
        buf = np.zeros((B, T), dtype=np.int32)
        buf[:b, :t] = ctx
        model.forward(torch.from_numpy(buf.reshape(-1)).cuda())
        return np.stack([model.logits(r * T + t - 1, 1)[0] for r in range(b)])

    return last_logits
