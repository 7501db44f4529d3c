"""Generation on the GPU through the C ABI: gpt2_op_sample against the
oracle's sampler, gpt2_forward_last against the full forward and the oracle,
gpt2_decode_step (the key/value cache) against the oracle's full forward,
and the library's generation loop against the oracle's loop on the same
uniforms (fp32 token for token, with and without the cache; bf16 greedy
within the bf16 logit error).

Where floating point decides the token (an inverse-CDF boundary), both sides
decide in their own precision; the comparisons assert equality only where the
oracle's cumulative sum is farther than 1e-5 (relative) from the draw, and
count the other cases, which the fixed inputs here do not produce."""
import numpy as np
import pytest
import torch

import synthdata
from decoder_only_transformer_06_b300 import gpt2
from decoder_only_transformer_06_b300.generate import draw_uniforms, generate
from oracle import CONFIGS
from oracle import gpt2_oracle as O

from gpu_helpers import dev, gpu_cfg
from test_generate import oracle_generate

pytestmark = pytest.mark.gpu


def _oracle_cdf(logits, temperature, top_k):
    """The oracle's cumulative weights per row (fp64) and the kept mask."""
    z = np.asarray(logits, np.float64) / temperature
    V = z.shape[1]
    keep = np.ones_like(z, dtype=bool)
    if top_k and 0 < top_k < V:
        kth = np.sort(z, axis=1)[:, V - top_k][:, None]
        keep = z >= kth
    w = np.where(keep, np.exp(z - z.max(axis=1, keepdims=True)), 0.0)
    return np.cumsum(w, axis=1), keep


def _margin(logits, temperature, top_k, u):
    """Relative distance of u*S to the nearest boundary of the oracle's CDF."""
    c, _ = _oracle_cdf(logits, temperature, top_k)
    tgt = np.asarray(u, np.float64)[:, None] * c[:, -1:]
    return (np.abs(c - tgt) / c[:, -1:]).min(axis=1)


def _check_valid(logits, temperature, top_k, u, tok, tol):
    """The device token is a kept entry whose CDF interval contains u*S up to
    tol*S in the oracle's fp64 arithmetic."""
    c, keep = _oracle_cdf(logits, temperature, top_k)
    rows = np.arange(c.shape[0])
    assert np.all(keep[rows, tok])
    S = c[:, -1]
    tgt = np.asarray(u, np.float64) * S
    lo = np.where(tok > 0, c[rows, np.maximum(tok - 1, 0)], 0.0)
    hi = c[rows, tok]
    assert np.all(lo - tol * S <= tgt) and np.all(tgt < hi + tol * S)


def _device_sample(logits, temperature, top_k, u):
    d = torch.from_numpy(np.ascontiguousarray(logits, dtype=np.float32)).cuda()
    du = torch.from_numpy(np.asarray(u, dtype=np.float32)).cuda()
    out = torch.empty(d.shape[0], dtype=torch.int32, device="cuda")
    gpt2.op_sample(d, temperature, top_k, du, out)
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.int64)


@pytest.mark.parametrize("V", [65, 50257])
def test_device_sampler_matches_the_oracle_sampler(V):
    """Same logits (fp32) and uniforms on both sides. Where the oracle's CDF
    boundary is farther than 2e-5 (relative) from the draw the tokens are
    identical; every device token is valid in the oracle's arithmetic up to
    that tolerance (fp32 cumulative sums over 50,257 entries carry ~5e-6)."""
    rng = np.random.default_rng(V)
    rows = 16
    logits = (2.0 * rng.standard_normal((rows, V))).astype(np.float32)
    logits[3, :7] = logits[3].max()                  # a tie at the maximum
    tol = 2e-5
    exact = 0
    for i, (temp, k) in enumerate(((0.8, 200), (1.0, None), (1.3, 5), (0.7, 1), (0.0, None))):
        u = (synthdata.uniforms(100 + i, np.arange(rows)) * 2 ** 24).astype(np.int64) * 2.0 ** -24
        got = _device_sample(logits, temp, k, u)
        want = O.sample_tokens(logits.astype(np.float64), temp, k, u)
        if temp <= 0:
            assert np.array_equal(got, want)
            continue
        safe = _margin(logits, temp, k, u) > tol
        assert np.array_equal(got[safe], want[safe]), (temp, k, got, want)
        exact += int(safe.sum())
        _check_valid(logits, temp, k, u, got, tol)
    assert exact >= 3 * rows                         # the top-k cases are all decided exactly


def test_device_sampler_appends_to_the_context_and_crops_it():
    V, rows, T = 65, 3, 8
    logits = torch.from_numpy(np.random.default_rng(1).standard_normal((rows, V)).astype(np.float32)).cuda()
    u = torch.full((rows,), 0.5, dtype=torch.float32, device="cuda")
    out = torch.empty(rows, dtype=torch.int32, device="cuda")
    base = np.arange(rows * T, dtype=np.int32).reshape(rows, T)
    ctx = torch.from_numpy(base.copy()).cuda()
    gpt2.op_sample(logits, 1.0, None, u, out, ctx=ctx, t=5)           # room left: written at 5
    tok = out.cpu().numpy()
    c = ctx.cpu().numpy()
    want = base.copy()
    want[:, 5] = tok
    assert np.array_equal(c, want)
    gpt2.op_sample(logits, 1.0, None, u, out, ctx=ctx, t=T)           # full: shift left, token at T-1
    c2 = ctx.cpu().numpy()
    want2 = np.concatenate([want[:, 1:], out.cpu().numpy()[:, None]], axis=1)
    assert np.array_equal(c2, want2)


@pytest.mark.parametrize("precision", [gpt2.GPT2_FP32, gpt2.GPT2_BF16])
def test_forward_last_matches_the_full_forward_and_the_oracle(precision):
    c = O.Config(n_layer=2, n_head=2, d_model=128, vocab_size=65, block_size=64, batch_size=3,
                 seq_len=64)
    m = gpt2.GPT2(gpu_cfg(c, precision), seed=9)
    params = O.init_params(c, 9)
    x, _ = synthdata.uniform_batch(65, c.batch_size, c.seq_len, 4)
    out = torch.empty(c.batch_size, c.vocab_size, dtype=torch.float32, device="cuda")
    _, ref, _ = O.forward(params, c, x)
    m.forward(dev(x))
    full = m.logits(0, c.batch_size * c.seq_len).reshape(c.batch_size, c.seq_len, -1)
    for t in (1, 17, 64):
        m.forward_last(dev(x), t, out)
        got = out.cpu().numpy()
        if precision == gpt2.GPT2_FP32:
            assert np.allclose(got, full[:, t - 1], rtol=1e-6, atol=1e-7)
            assert np.allclose(got, ref[:, t - 1], rtol=1e-4, atol=1e-5)
        else:
            # the full forward keeps bf16 logits; the last-position head keeps fp32
            assert np.allclose(got, full[:, t - 1], rtol=2 ** -7, atol=1e-3)
            err = np.linalg.norm(got - ref[:, t - 1]) / np.linalg.norm(ref[:, t - 1])
            assert err < 2e-2, err
    m.close()


@pytest.mark.parametrize("kv_cache", [True, False])
def test_library_generation_matches_the_oracle_fp32(kv_cache):
    """fp32-math mode: the library's loop (device forward_last or the
    key/value-cache step, + sampler) against the oracle's loop (a full forward
    per token) on the same uniforms, greedy and sampled (top-k 5, temperature
    0.8), past the block size (the context is cropped, after which the cached
    positions no longer hold and the loop runs the full forward again)."""
    c = CONFIGS["tiny"]
    m = gpt2.GPT2(gpu_cfg(c, gpt2.GPT2_FP32), seed=4)
    params = O.init_params(c, 4)
    prompt = np.random.default_rng(9).integers(0, c.vocab_size, size=(2, 5))
    n = c.block_size + 4
    u = np.stack([draw_uniforms(3, s, c.batch_size) for s in range(n)])
    for top_k, temp in ((1, 1.0), (5, 0.8), (None, 0.0)):
        a = generate(m, prompt, n, temperature=temp, top_k=top_k, uniforms=u, kv_cache=kv_cache)
        b = oracle_generate(params, c, prompt, n, temp, top_k, u)
        assert np.array_equal(a, b), (top_k, temp)
    m.close()


@pytest.mark.parametrize("precision", [gpt2.GPT2_FP32, gpt2.GPT2_BF16])
def test_decode_step_matches_the_oracle(precision):
    """A chain of cached steps after one forward_last: the logits of position
    t-1 for t = t0+1 .. T (the last step fills the block) against the
    oracle's full forward on the same context, and against forward_last on
    that context afterwards (same library, no cache)."""
    c = O.Config(n_layer=2, n_head=2, d_model=128, vocab_size=65, block_size=64, batch_size=3,
                 seq_len=64)
    m = gpt2.GPT2(gpu_cfg(c, precision), seed=9)
    params = O.init_params(c, 9)
    x, _ = synthdata.uniform_batch(65, c.batch_size, c.seq_len, 5)
    _, ref, _ = O.forward(params, c, x)
    t0 = 57
    out = torch.empty(c.batch_size, c.vocab_size, dtype=torch.float32, device="cuda")
    d_x = dev(x).view(c.batch_size, c.seq_len)
    m.forward_last(d_x.reshape(-1), t0, out)
    got = {}
    for t in range(t0 + 1, c.seq_len + 1):
        tok = d_x[:, t - 1].contiguous()
        m.decode_step(tok, t, out)
        got[t] = out.cpu().numpy().copy()
    for t, g in got.items():
        m.forward_last(d_x.reshape(-1), t, out)
        nocache = out.cpu().numpy()
        want = ref[:, t - 1]
        if precision == gpt2.GPT2_FP32:
            assert np.allclose(g, want, rtol=1e-4, atol=1e-5), t
            assert np.allclose(g, nocache, rtol=1e-5, atol=1e-5), t
        else:
            err = np.linalg.norm(g - want) / np.linalg.norm(want)
            assert err < 2e-2, (t, err)
            err2 = np.linalg.norm(g - nocache) / np.linalg.norm(nocache)
            assert err2 < 1e-2, (t, err2)
    m.close()


def test_decode_step_needs_the_cached_positions():
    c = CONFIGS["tiny"]
    m = gpt2.GPT2(gpu_cfg(c, gpt2.GPT2_FP32), seed=2)
    x, y = synthdata.uniform_batch(c.vocab_size, c.batch_size, c.seq_len, 6)
    out = torch.empty(c.batch_size, c.vocab_size, dtype=torch.float32, device="cuda")
    d_x = dev(x)
    tok = d_x.view(c.batch_size, c.seq_len)[:, 0].contiguous()
    with pytest.raises(gpt2.GPT2Error) as e:
        m.decode_step(tok, 2, out)                     # nothing cached yet
    assert e.value.code == gpt2.GPT2_ESTATE
    m.decode_step(tok, 1, out)                         # position 0 needs no cache
    m.forward_last(d_x, 5, out)
    m.decode_step(d_x.view(c.batch_size, c.seq_len)[:, 5].contiguous(), 6, out)
    m.forward(d_x, dev(y))                             # a training forward overwrites the cache
    with pytest.raises(gpt2.GPT2Error) as e:
        m.decode_step(tok, 7, out)
    assert e.value.code == gpt2.GPT2_ESTATE
    with pytest.raises(gpt2.GPT2Error) as e:
        m.decode_step(tok, c.seq_len + 1, out)
    assert e.value.code == gpt2.GPT2_EINVAL
    # an id outside the vocabulary is clamped and reported by the next synchronising call
    m.forward_last(d_x, 5, out)
    bad = torch.full((c.batch_size,), c.vocab_size + 3, dtype=torch.int32, device="cuda")
    m.decode_step(bad, 6, out)
    with pytest.raises(gpt2.GPT2Error) as e:
        m.sync()
    assert e.value.code == gpt2.GPT2_ERANGE
    m.close()


def test_library_generation_bf16():
    """bf16 mode. Greedy: at every step the library's token is, on the
    oracle's logits for the library's own context, within 0.01 of the
    oracle's best (the bf16 error of these logits is about 1e-3). Sampled: on
    the library's own logits of each step, the device sampler and the
    oracle's sampler choose the same token."""
    c = O.Config(n_layer=2, n_head=2, d_model=128, vocab_size=65, block_size=64, batch_size=2,
                 seq_len=64)
    m = gpt2.GPT2(gpu_cfg(c, gpt2.GPT2_BF16), seed=12)
    params = O.init_params(c, 12)
    prompt = np.random.default_rng(5).integers(0, c.vocab_size, size=(2, 6))
    n = 20
    a = generate(m, prompt, n, temperature=0.0)
    for s in range(n):
        ctx = a[:, : prompt.shape[1] + s][:, -c.block_size:]
        _, logits, _ = O.forward(params, c, ctx)
        last = logits[:, -1, :]
        picked = last[np.arange(2), a[:, prompt.shape[1] + s]]
        assert np.all(picked >= last.max(axis=1) - 0.01), s
    # sampled: the device sampler on the library's own bf16-model logits
    d_ctx = torch.zeros(c.batch_size * c.seq_len, dtype=torch.int32, device="cuda")
    d_ctx.view(c.batch_size, c.seq_len)[:, :6] = torch.from_numpy(prompt.astype(np.int32)).cuda()
    d_logits = torch.empty(c.batch_size, c.vocab_size, dtype=torch.float32, device="cuda")
    m.forward_last(d_ctx, 6, d_logits)
    lg = d_logits.cpu().numpy()
    for i in range(10):
        u = draw_uniforms(40 + i, 0, c.batch_size)
        got = _device_sample(lg, 0.9, 10, u)
        want = O.sample_tokens(lg.astype(np.float64), 0.9, 10, u.astype(np.float64))
        assert np.all(_margin(lg, 0.9, 10, u) > 1e-5)
        assert np.array_equal(got, want)
    m.close()
