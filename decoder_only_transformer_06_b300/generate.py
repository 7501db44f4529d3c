"""Sampling from a trained model on the GPU, as the pages' generate loop does it
("Let's reproduce GPT-2", 00:37:02 the sampling loop; nanoGPT guide, sample.py):
crop the context to the block size, take the logits of the last position,
divide by the temperature, keep the top k, softmax, draw one token, append,
repeat. There is no KV cache: every new token runs the forward again on the
whole context.

Every step runs in the library: gpt2_forward_last (the blocks on the [B, T]
context, the LM head on position t-1 only) or, with the key/value cache,
gpt2_decode_step (position t-1 alone), and gpt2_op_sample (temperature,
top-k, softmax, inverse-CDF draw, and the append to the context, shifting it
left once it holds T tokens). The host only draws the uniforms the sampler
consumes and copies the new tokens back at the end. The pages have no
key/value cache: it changes the work per token, not the result.

Uniforms: u[step, row] = the top 24 bits of output number step*B + row of a
SplitMix64 stream (Steele, Lea & Flood, OOPSLA 2014) started at the seed,
times 2^-24 (exact in fp32, in [0, 1)). Callers may pass their own instead.
"""
from __future__ import annotations

import numpy as np

_GAMMA = 0x9E3779B97F4A7C15
_MASK = (1 << 64) - 1


def draw_uniforms(seed: int, step: int, rows: int) -> np.ndarray:
    """fp32 [rows]: u for one generation step (see the module docstring)."""
    out = np.empty(rows, dtype=np.float32)
    for r in range(rows):
        z = (seed + (step * rows + r + 1) * _GAMMA) & _MASK
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK
        z ^= z >> 31
        out[r] = (z >> 40) * (2.0 ** -24)
    return out


def generate(model, prompt, max_new_tokens, temperature=1.0, top_k=None, seed=0, uniforms=None,
             kv_cache=True):
    """Extend every row of `prompt` (int [b, t0], b <= B, t0 >= 1) by
    max_new_tokens tokens sampled by the library's model (a gpt2.GPT2 of batch
    B and sequence length T, the block size of the loop). temperature <= 0
    decodes greedily. uniforms: optional fp32 [max_new_tokens, B] to use
    instead of the seeded draws. kv_cache: after the first full forward, each
    new position runs alone against the cached keys and values
    (gpt2_decode_step) until the context is full; once the crop to T shifts
    the positions, the full forward runs again. Returns int64
    [b, t0 + max_new_tokens]."""
    import torch
    from . import gpt2

    idx = np.asarray(prompt, dtype=np.int64)
    B, T, V = model.cfg.batch_size, model.cfg.seq_len, model.cfg.vocab_size
    if idx.ndim != 2 or idx.shape[1] < 1 or idx.shape[0] > B:
        raise ValueError(f"prompt must be [b <= {B}, t0 >= 1]")
    b, t0 = idx.shape
    if uniforms is not None:
        uniforms = np.asarray(uniforms, dtype=np.float32)
        if uniforms.shape != (max_new_tokens, B):
            raise ValueError(f"uniforms must be [{max_new_tokens}, {B}]")
    t = min(t0, T)
    ctx = np.zeros((B, T), dtype=np.int32)
    ctx[:b, :t] = idx[:, t0 - t:]
    stream = model.stream
    with torch.cuda.stream(stream):
        d_ctx = torch.from_numpy(ctx).cuda()
        d_logits = torch.empty(B, V, dtype=torch.float32, device="cuda")
        d_new = torch.empty(max_new_tokens, B, dtype=torch.int32, device="cuda")
        u_all = uniforms if uniforms is not None else np.stack(
            [draw_uniforms(seed, s, B) for s in range(max_new_tokens)]) if max_new_tokens else \
            np.zeros((0, B), np.float32)
        d_u = torch.from_numpy(np.ascontiguousarray(u_all)).cuda()
        full = True                  # the cache does not hold positions 0..t-2
        for s in range(max_new_tokens):
            if full or not kv_cache:
                model.forward_last(d_ctx.view(-1), t, d_logits)
            else:
                model.decode_step(d_new[s - 1], t, d_logits)
            gpt2.op_sample(d_logits, temperature, top_k, d_u[s], d_new[s], ctx=d_ctx, t=t,
                           stream=stream)
            full = t == T                # a full context was shifted left by the append
            t = min(t + 1, T)
        new = d_new.cpu().numpy()
    return np.concatenate([idx, new[:, :b].T.astype(np.int64)], axis=1)
