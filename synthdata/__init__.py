"""Seeded synthetic token streams for the GPT-2 training step.

This module is the only code shared by the CUDA path's tests/bench and the
oracle. It holds no arithmetic of the model: it only draws token ids.

The corpora the pages train on (FineWeb-Edu, OpenWebText, Tiny Shakespeare;
"Let's reproduce GPT-2 (124M)" sections 03:10:21 and 02:26:21, nanoGPT guide
"Deep dive 3: the data pipeline") are not available, so these streams stand in
for them with the same shapes:

* ``zipf_batch``     -- GPT-2 BPE-sized vocabularies: ids drawn i.i.d. from a
  Zipf(s) law p(r) ~ r^-s over ranks r = 1..V, id = r - 1.
* ``markov_batch``   -- the 65-symbol character corpus: an order-1 Markov
  chain (Metropolis, uniform proposal) whose stationary law is Zipf(s).
* ``uniform_batch``  -- ids uniform in [0, V).

Every batch follows the pages' windowing (nanoGPT guide, Part IV Stage 3):
each of the B rows is an independent window of T+1 draws s[0..T]; inputs are
x = s[0:T] and targets y = s[1:T+1].

Randomness is counter based: the n-th draw of a stream with seed S is
SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014) advanced n+1 times from state S, mapped to a double
in [0,1) by its top 53 bits.
"""
from __future__ import annotations

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def splitmix64(state: int, counters: np.ndarray) -> np.ndarray:
    """Output number ``counters`` (0-based) of a SplitMix64 stream started at ``state``."""
    with np.errstate(over="ignore"):
        z = np.uint64(state & 0xFFFFFFFFFFFFFFFF) + (counters.astype(np.uint64) + np.uint64(1)) * _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def uniforms(state: int, counters: np.ndarray) -> np.ndarray:
    """Doubles in [0, 1) from the top 53 bits of the stream outputs."""
    return (splitmix64(state, counters) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def zipf_pmf(V: int, s: float = 1.1) -> np.ndarray:
    r = np.arange(1, V + 1, dtype=np.float64)
    w = r ** (-s)
    return w / w.sum()


def _inverse_cdf(cdf: np.ndarray, u: np.ndarray) -> np.ndarray:
    idx = np.searchsorted(cdf, u, side="right")
    return np.minimum(idx, cdf.shape[0] - 1)


def _split(s: np.ndarray):
    return (np.ascontiguousarray(s[:, :-1]).astype(np.int32),
            np.ascontiguousarray(s[:, 1:]).astype(np.int32))


def zipf_batch(V: int, B: int, T: int, seed: int, s: float = 1.1):
    """(x, y) int32 [B, T]: i.i.d. Zipf(s) ids over [0, V)."""
    cdf = np.cumsum(zipf_pmf(V, s))
    n = np.arange(B * (T + 1), dtype=np.uint64)
    seq = _inverse_cdf(cdf, uniforms(seed, n)).reshape(B, T + 1)
    return _split(seq)


def uniform_batch(V: int, B: int, T: int, seed: int):
    """(x, y) int32 [B, T]: ids uniform in [0, V)."""
    n = np.arange(B * (T + 1), dtype=np.uint64)
    seq = np.minimum((uniforms(seed, n) * V).astype(np.int64), V - 1).reshape(B, T + 1)
    return _split(seq)


def markov_batch(V: int, B: int, T: int, seed: int, s: float = 1.1):
    """(x, y) int32 [B, T] from an order-1 Markov chain with Zipf(s) stationary law.

    Metropolis chain: from state i propose j uniform over [0, V), accept with
    probability min(1, pi_j / pi_i). Detailed balance holds, so pi is
    stationary; the first symbol of each row is drawn from pi.
    """
    pi = zipf_pmf(V, s)
    cdf = np.cumsum(pi)
    # counters: row b uses [b * 2(T+1), (b+1) * 2(T+1)); two draws per position
    base = np.arange(B, dtype=np.uint64) * np.uint64(2 * (T + 1))
    seq = np.empty((B, T + 1), dtype=np.int64)
    seq[:, 0] = _inverse_cdf(cdf, uniforms(seed, base))
    for t in range(1, T + 1):
        up = uniforms(seed, base + np.uint64(2 * t))
        ua = uniforms(seed, base + np.uint64(2 * t + 1))
        prop = np.minimum((up * V).astype(np.int64), V - 1)
        cur = seq[:, t - 1]
        accept = ua < np.minimum(1.0, pi[prop] / pi[cur])
        seq[:, t] = np.where(accept, prop, cur)
    return _split(seq)


# Named stand-ins for the workloads, keyed like the configurations they serve.
def batch_for(kind: str, V: int, B: int, T: int, seed: int):
    if kind == "zipf":
        return zipf_batch(V, B, T, seed)
    if kind == "markov":
        return markov_batch(V, B, T, seed)
    if kind == "uniform":
        return uniform_batch(V, B, T, seed)
    raise ValueError(f"unknown token stream kind {kind!r}")
