"""Model-level parity: the library's forward / backward / step against the
oracle on the same seeded inputs, through the C ABI.

Tolerances:
  fp32-math mode: loss and every gradient within 1e-4 relative (per-tensor L2).
  bf16 mode: loss within 5e-3 relative; per-tensor gradient relative L2 <= 2e-2
  and cosine >= 0.999; after AdamW, parameters within 1e-3 absolute.
Post-AdamW parameters are checked two ways. (1) The optimizer in isolation:
the oracle's clip + AdamW fed the GPU's own gradients reproduces the GPU's
parameters within 1e-6 absolute. (2) End to end (see adamw_param_check): a
first Adam step moves every element by ~lr whatever |g|, so the 1e-3 bound
applies where the two gradients agree in sign (fp32: 1e-6 where also
|g| >= 100 eps); no element with a large gradient may flip sign; every
element stays within 2 lr (plus decay) of the oracle.
"""
import math

import numpy as np
import pytest
import torch

import synthdata
from decoder_only_transformer_06_b300 import gpt2
from oracle import CONFIGS
from oracle import gpt2_oracle as O

from gpu_helpers import adamw_param_check, cosine, dev, gpu_cfg, oracle_adamw_on, oracle_cfg, rel_l2

pytestmark = pytest.mark.gpu


def _compare_step(ocfg, precision, kind, seed=1337, data_seed=42, lr=1e-3, ignore=None):
    m = gpt2.GPT2(gpu_cfg(ocfg, precision), seed=seed)
    tr = O.Trainer(ocfg, seed)
    # independent inits agree (bit-exact up to a rare fp32 ulp, see test_abi)
    for name in m.names:
        assert np.allclose(m.get(name), tr.params[name], rtol=2 ** -23, atol=0), name
    x, y = synthdata.batch_for(kind, ocfg.vocab_size, ocfg.batch_size, ocfg.seq_len, data_seed)
    if ignore is not None:
        y = y.copy()
        y[ignore] = -1
    loss = m.forward(dev(x), dev(y))
    lo, _ = tr.forward(x, y)
    m.backward()
    tr.backward()
    g_gpu = m.state(gpt2.GPT2_GRAD)
    p0 = {n: a.copy() for n, a in tr.params.items()}
    norm = m.step(lr=lr)
    p_gpu = m.state(gpt2.GPT2_PARAM)
    g_orc = {n: a.copy() for n, a in tr.grads.items()}
    tn = tr.step(lr=lr)
    out = dict(loss=(loss, lo), norm=(norm, tn), g_gpu=g_gpu, g_orc=g_orc, p_gpu=p_gpu,
               p_orc=tr.params, m=m, tr=tr, V=ocfg.vocab_size,
               p_iso=oracle_adamw_on(p0, g_gpu, lr))
    return out


def _check_isolated_adamw(r):
    for n, p in r["p_iso"].items():
        d = float(np.abs(r["p_gpu"][n] - p).max())
        assert d < 1e-6, (n, d)


def _check_fp32(r):
    loss, lo = r["loss"]
    assert abs(loss - lo) / abs(lo) < 1e-4
    for n, g in r["g_orc"].items():
        e = rel_l2(r["g_gpu"][n], g)
        assert e < 1e-4, (n, e)
    assert abs(r["norm"][0] - r["norm"][1]) / r["norm"][1] < 1e-4
    _check_isolated_adamw(r)
    coef = min(1.0, 1.0 / (r["norm"][1] + 1e-6))       # clip 1.0
    for n in r["p_orc"]:
        d, flips, _ = adamw_param_check(r["p_gpu"][n], r["p_orc"][n], r["g_gpu"][n],
                                        r["g_orc"][n], fp32=True, coef=coef)
        assert d < 1e-6, (n, d)
        assert flips == 0, (n, flips)


def _check_bf16(r):
    loss, lo = r["loss"]
    assert abs(loss - lo) / abs(lo) < 5e-3, (loss, lo)
    for n, g in r["g_orc"].items():
        if not np.any(g):
            assert not np.any(r["g_gpu"][n]), n
            continue
        e, c = rel_l2(r["g_gpu"][n], g), cosine(r["g_gpu"][n], g)
        assert e <= 2e-2 and c >= 0.999, (n, e, c)
    assert abs(r["norm"][0] - r["norm"][1]) / r["norm"][1] < 2e-2
    _check_isolated_adamw(r)
    for n in r["p_orc"]:
        d, flips, dmax = adamw_param_check(r["p_gpu"][n], r["p_orc"][n], r["g_gpu"][n],
                                           r["g_orc"][n], fp32=False)
        assert d <= 1e-3, (n, d)
        assert flips <= max(2, r["p_orc"][n].size // 100000), (n, flips)
        assert dmax <= 2.2e-3, (n, dmax)      # 2 lr (+ decay) for any element


def _pad_rows_zero(r):
    V = r["V"]
    assert np.all(r["g_gpu"]["wte"][V:] == 0.0)
    assert np.all(r["g_orc"]["wte"][V:] == 0.0)


def test_tiny_fp32_one_full_step():
    """Tiny GPT (2 layers, 4 heads, d=64, V=65, T=64, B=4), fp32-math mode."""
    r = _compare_step(CONFIGS["tiny"], gpt2.GPT2_FP32, "uniform")
    _check_fp32(r)
    _pad_rows_zero(r)


def test_tiny_fp32_ignore_index():
    r = _compare_step(CONFIGS["tiny"], gpt2.GPT2_FP32, "uniform",
                      ignore=(np.array([0, 1, 3, 3]), np.array([5, 63, 0, 1])))
    _check_fp32(r)


def test_char_bf16_one_step_reduced_batch():
    """Character model (6 layers, d=384, T=256) at B=8, bf16 mode."""
    r = _compare_step(oracle_cfg(CONFIGS["char"], batch_size=8), gpt2.GPT2_BF16, "markov")
    _check_bf16(r)
    _pad_rows_zero(r)


def test_char_fp32_one_step_reduced_batch():
    r = _compare_step(oracle_cfg(CONFIGS["char"], batch_size=4), gpt2.GPT2_FP32, "markov")
    _check_fp32(r)


def test_bf16_ragged_sequence_and_small_width():
    """T not a multiple of the 64-row tiles, d=128 (2 heads of 64), V=65."""
    c = O.Config(n_layer=2, n_head=2, d_model=128, vocab_size=65, block_size=100, batch_size=3,
                 seq_len=100)
    r = _compare_step(c, gpt2.GPT2_BF16, "uniform",
                      ignore=(np.array([0, 2]), np.array([99, 17])))
    _check_bf16(r)


def test_bf16_single_token_sequences():
    c = O.Config(n_layer=1, n_head=1, d_model=64, vocab_size=65, block_size=8, batch_size=5,
                 seq_len=1)
    r = _compare_step(c, gpt2.GPT2_BF16, "uniform")
    _check_bf16(r)


@pytest.mark.slow
def test_gpt2_124m_bf16_one_step_batch2():
    """GPT-2 124M at B=2, T=1024 (the full-width model; oracle in fp64)."""
    r = _compare_step(oracle_cfg(CONFIGS["gpt2_124m"], batch_size=2), gpt2.GPT2_BF16, "zipf",
                      lr=6e-4)
    _check_bf16(r)
    _pad_rows_zero(r)


@pytest.mark.slow
def test_char_bf16_loss_trajectory():
    """The character model of the pages' configuration (6 layers, 6 heads,
    d=384, T=256, Markov-chain tokens) at B=16, 20 AdamW steps at lr 1e-3 on
    fresh batches, every step checked on the same parameters: before each step
    the oracle takes the library's current parameters, so the library's loss
    is held to the stated one-step bound (5e-3 relative) at each of 20 points
    along its own bf16 trajectory, its gradients to the bf16 gradient bounds
    (every fifth step), and its clip + AdamW update, given its own gradients
    and moments, to the oracle's update of them within 1e-6.

    A free-running fp64 run from the same init is compared too, but only
    reported: the two runs separate step by step (an Adam step moves every
    element by about lr whatever |g|, so elements whose tiny gradient differs
    in sign move apart by 2 lr per step; measured on B300 the curves differ by
    about 6% after 17 steps), so the one-step bound does not apply to them."""
    c = oracle_cfg(CONFIGS["char"], batch_size=16)
    m = gpt2.GPT2(gpu_cfg(c, gpt2.GPT2_BF16), seed=3)
    synced = O.Trainer(c, 3)         # re-synced to the library's parameters each step
    free = O.Trainer(c, 3)           # free-running fp64 trajectory (reported only)
    worst_step, worst_curve = 0.0, 0.0
    for step in range(20):
        x, y = synthdata.markov_batch(65, c.batch_size, c.seq_len, 100 + step)
        p0 = m.state(gpt2.GPT2_PARAM)
        for n in synced.params:
            synced.params[n] = p0[n].astype(np.float64)
        m.zero_grad()
        synced.zero_grad()
        free.zero_grad()
        loss = m.forward(dev(x), dev(y))
        lo, _ = synced.forward(x, y)
        lf, _ = free.forward(x, y)
        rel = abs(loss - lo) / lo
        worst_step = max(worst_step, rel)
        assert rel < 5e-3, (step, loss, lo)
        worst_curve = max(worst_curve, abs(loss - lf) / lf)
        m.backward()
        synced.backward()
        free.backward()
        g = m.state(gpt2.GPT2_GRAD)
        if step % 5 == 4:
            for n, ref in synced.grads.items():
                if not np.any(ref):
                    continue
                e, cs = rel_l2(g[n], ref), cosine(g[n], ref)
                assert e <= 2e-2 and cs >= 0.999, (step, n, e, cs)
        mom = (m.state(gpt2.GPT2_ADAM_M), m.state(gpt2.GPT2_ADAM_V))
        m.step(lr=1e-3)
        free.step(lr=1e-3)
        # the library's update in isolation: the oracle's clip + AdamW (step
        # t = step + 1) applied to the library's gradients and moments
        p1 = m.state(gpt2.GPT2_PARAM)
        gg = {n: a.astype(np.float64) for n, a in g.items()}
        O.clip_grads(gg, 1.0)
        for n in p1:
            ref = p0[n].astype(np.float64)
            mm, vv = mom[0][n].astype(np.float64), mom[1][n].astype(np.float64)
            O.adamw_update(ref, gg[n], mm, vv, step + 1, 1e-3, 0.9, 0.95, 1e-8, 0.1, ref.ndim >= 2)
            d = float(np.abs(p1[n] - ref).max())
            assert d < 1e-6, (step, n, d)
    print(f"char bf16 20 steps: worst same-parameter loss difference {worst_step:.2e}; "
          f"free-running curves differ by up to {worst_curve:.2e}")


@pytest.mark.slow
def test_full_vocabulary_fp32_embedding_gradients():
    """fp32-math mode at GPT-2's vocabulary and sequence length with Zipf-hot
    ids (4,096 rows): the embedding backward's token sort runs both 8-bit
    passes of the radix sort and the hot tokens' segments span many chunks
    (the carry pass); every gradient, wte and wpe included, within 1e-4 of the
    oracle."""
    c = O.Config(n_layer=1, n_head=2, d_model=64, vocab_size=50257, padded_vocab=50304,
                 block_size=1024, batch_size=4, seq_len=1024)
    r = _compare_step(c, gpt2.GPT2_FP32, "zipf", lr=6e-4)
    _check_fp32(r)
    _pad_rows_zero(r)


def test_gpt2_width_full_batch_bf16_gradients():
    """The benchmark's batch shape (B=16, T=1024: 16,384 rows) at GPT-2 width
    and full vocabulary with two layers: every gradient against the oracle.
    Reaches the row-count-dependent paths at full size: cross-entropy over
    16,384 rows of 50,304 columns, the token sort of the embedding backward
    with the Zipf-hot ids, the attention work lists of 16 x 12 heads."""
    c = oracle_cfg(CONFIGS["gpt2_124m"], n_layer=2)
    r = _compare_step(c, gpt2.GPT2_BF16, "zipf", lr=6e-4)
    _check_bf16(r)
    _pad_rows_zero(r)


@pytest.mark.slow
def test_gpt2_medium_width_bf16_one_step():
    """The 24-layer configuration's widths (d=1024, 16 heads of 64, MLP 4096,
    vocabulary 50304) with two layers at B=2, T=1024: one full step."""
    c = oracle_cfg(CONFIGS["gpt2_24l_1024d"], n_layer=2, batch_size=2)
    r = _compare_step(c, gpt2.GPT2_BF16, "zipf", lr=6e-4)
    _check_bf16(r)
    _pad_rows_zero(r)


@pytest.mark.parametrize("precision", [gpt2.GPT2_FP32, gpt2.GPT2_BF16])
def test_grad_accumulation_matches_the_oracle(precision):
    """Four micro-steps of B=2 with grad_accum_steps=4 (sotaaz Section 3:
    each micro-batch loss divided by the micro-batch count; gradients add up
    across backward calls) against the oracle's Trainer over the same four
    micro-batches: accumulated gradients, the clipped norm and the update."""
    base = oracle_cfg(CONFIGS["char"], n_layer=2, batch_size=2, grad_accum_steps=4)
    m = gpt2.GPT2(gpu_cfg(base, precision), seed=8)
    tr = O.Trainer(base, 8)
    for i in range(4):
        x, y = synthdata.markov_batch(65, base.batch_size, base.seq_len, 300 + i)
        loss = m.forward(dev(x), dev(y))
        lo, _ = tr.forward(x, y)
        assert abs(loss - lo) / lo < (1e-4 if precision == gpt2.GPT2_FP32 else 5e-3), (i, loss, lo)
        m.backward()
        tr.backward()
    g_gpu = m.state(gpt2.GPT2_GRAD)
    g_orc = {n: a.copy() for n, a in tr.grads.items()}
    p0 = {n: a.copy() for n, a in tr.params.items()}
    norm = m.step(lr=1e-3)
    tn = tr.step(lr=1e-3)
    r = dict(loss=(loss, lo), norm=(norm, tn), g_gpu=g_gpu, g_orc=g_orc,
             p_gpu=m.state(gpt2.GPT2_PARAM), p_orc=tr.params, V=base.vocab_size,
             p_iso=oracle_adamw_on(p0, g_gpu, 1e-3))
    if precision == gpt2.GPT2_FP32:
        _check_fp32(r)
    else:
        _check_bf16(r)
    _pad_rows_zero(r)


def test_fp32_consecutive_steps_track_the_oracle():
    """Three training steps in a row, zero_grad after each step. The library
    runs each step's AdamW on its second stream while the next forward waits
    for every parameter group just before using it, and queues zero_grad behind
    that update: a layer that read a parameter before its update, or gradients
    not cleared before the next backward, would move the next step's loss by far
    more than the fp32 tolerance."""
    c = CONFIGS["tiny"]
    m = gpt2.GPT2(gpu_cfg(c, gpt2.GPT2_FP32), seed=11)
    tr = O.Trainer(c, 11)
    for step in range(3):
        x, y = synthdata.uniform_batch(65, c.batch_size, c.seq_len, 500 + step)
        loss = m.forward(dev(x), dev(y))
        lo, _ = tr.forward(x, y)
        assert abs(loss - lo) / lo < 1e-4, (step, loss, lo)
        m.backward()
        tr.backward()
        m.step(lr=3e-3)
        tr.step(lr=3e-3)
        m.zero_grad()
        tr.zero_grad()
    # after the last update: parameters (read through a copy, which waits for
    # the pending update) close to the oracle's. An Adam step moves an element
    # by about lr whatever |g|, so an element whose tiny gradient has the other
    # sign may differ by up to 2 lr per step: 6 lr after three steps.
    p = m.state(gpt2.GPT2_PARAM)
    for n, a in tr.params.items():
        assert float(np.abs(p[n] - a).max()) <= 6 * 3e-3, n
        assert rel_l2(p[n], a) < 1e-2, (n, rel_l2(p[n], a))
    g = m.state(gpt2.GPT2_GRAD)
    assert all(not np.any(v) for v in g.values())


def test_grad_accumulation_matches_one_big_batch():
    base = CONFIGS["tiny"]
    x, y = synthdata.uniform_batch(65, 8, base.seq_len, 9)
    big = gpt2.GPT2(gpu_cfg(oracle_cfg(base, batch_size=8), gpt2.GPT2_FP32), seed=5)
    big.forward(dev(x), dev(y))
    big.backward()
    acc = gpt2.GPT2(gpu_cfg(oracle_cfg(base, batch_size=2, grad_accum_steps=4), gpt2.GPT2_FP32),
                    seed=5)
    for i in range(4):
        acc.forward(dev(x[2 * i:2 * i + 2]), dev(y[2 * i:2 * i + 2]))
        acc.backward()
    gb, ga = big.state(gpt2.GPT2_GRAD), acc.state(gpt2.GPT2_GRAD)
    for n in gb:
        assert rel_l2(ga[n], gb[n]) < 1e-5, n


def test_async_loss_read_matches_the_synchronous_one():
    """gpt2_get_loss_async enqueues the copy on the model's stream: after a
    sync the pinned host value equals gpt2_get_loss's, step after step."""
    c = CONFIGS["tiny"]
    m = gpt2.GPT2(gpu_cfg(c, gpt2.GPT2_FP32), seed=3)
    h = torch.zeros(3, dtype=torch.float32).pin_memory()
    for i in range(3):
        x, y = synthdata.uniform_batch(c.vocab_size, c.batch_size, c.seq_len, 20 + i)
        m.forward(dev(x), dev(y), sync_loss=False)
        m.loss_async(h[i:i + 1])
        m.backward()
        m.step(lr=1e-3, sync_norm=False)
        m.zero_grad()
        m.sync()
        assert h[i].item() == m.loss()
    m.close()


def test_runs_are_bit_reproducible():
    c = oracle_cfg(CONFIGS["char"], batch_size=4, n_layer=2)
    x, y = synthdata.markov_batch(65, c.batch_size, c.seq_len, 1)
    outs = []
    for _ in range(2):
        m = gpt2.GPT2(gpu_cfg(c, gpt2.GPT2_BF16), seed=1)
        loss = m.forward(dev(x), dev(y))
        m.backward()
        outs.append((loss, m.state(gpt2.GPT2_GRAD)))
        m.close()
    assert outs[0][0] == outs[1][0]
    for n in outs[0][1]:
        assert np.array_equal(outs[0][1][n], outs[1][1][n]), n


def test_errors_are_reported_and_recoverable():
    c = CONFIGS["tiny"]
    m = gpt2.GPT2(gpu_cfg(c, gpt2.GPT2_FP32), seed=1)
    with pytest.raises(gpt2.GPT2Error) as e:
        m.backward()
    assert e.value.code == gpt2.GPT2_ESTATE
    x, y = synthdata.uniform_batch(65, c.batch_size, c.seq_len, 2)
    bad = x.copy()
    bad[0, 3] = 70000
    with pytest.raises(gpt2.GPT2Error) as e:
        m.forward(dev(bad), dev(y))
    assert e.value.code == gpt2.GPT2_ERANGE
    bady = y.copy()
    bady[1, 1] = -5
    with pytest.raises(gpt2.GPT2Error) as e:
        m.forward(dev(x), dev(bady))
    assert e.value.code == gpt2.GPT2_ERANGE
    loss = m.forward(dev(x), dev(y))          # the model stays usable
    assert math.isfinite(loss)
    m.backward()
    m.step(lr=1e-3)


def test_nonfinite_gradient_skips_the_update():
    c = CONFIGS["tiny"]
    m = gpt2.GPT2(gpu_cfg(c, gpt2.GPT2_FP32), seed=1)
    x, y = synthdata.uniform_batch(65, c.batch_size, c.seq_len, 2)
    m.forward(dev(x), dev(y))
    m.backward()
    g = m.get("lnf.b", gpt2.GPT2_GRAD)
    g[0] = np.nan
    m.set("lnf.b", g, gpt2.GPT2_GRAD)
    before = m.state()
    with pytest.raises(gpt2.GPT2Error) as e:
        m.step(lr=1e-3)
    assert e.value.code == gpt2.GPT2_ENONFINITE
    after = m.state()
    for n in before:
        assert np.array_equal(before[n], after[n], equal_nan=True), n
    m.zero_grad()
    m.forward(dev(x), dev(y))
    m.backward()
    assert math.isfinite(m.step(lr=1e-3))


def test_num_params_matches_pages_through_the_library():
    m = gpt2.GPT2(gpu_cfg(CONFIGS["gpt2_124m"], gpt2.GPT2_BF16, batch_size=1, seq_len=64), seed=1)
    assert m.num_params(include_wpe=False) == 123_653_376
    assert m.num_params() == 124_439_808
    assert m.num_params(padded=True) == 124_475_904


@pytest.mark.slow
def test_gpt2_124m_full_size_sampled_rows():
    """The benchmark's workload (B=16, T=1024, bf16): per-row losses of two
    sampled sequences against the oracle run on those sequences alone, the
    mean loss against the sampled mean, and a finite clipped step."""
    c = CONFIGS["gpt2_124m"]
    m = gpt2.GPT2(gpu_cfg(c, gpt2.GPT2_BF16), seed=1337)
    x, y = synthdata.zipf_batch(c.vocab_size, c.batch_size, c.seq_len, 1337)
    loss = m.forward(dev(x), dev(y))
    rows = m.row_losses().reshape(c.batch_size, c.seq_len)
    params = O.init_params(c, 1337)
    one = oracle_cfg(c, batch_size=1)
    for b in (0, 11):
        lo, _, cache = O.forward(params, one, x[b:b + 1], y[b:b + 1])
        ref_rows = cache["row_loss"][0]
        assert np.abs(rows[b] - ref_rows).max() < 0.05
        assert abs(rows[b].mean() - lo) / lo < 5e-3
    assert abs(loss - rows.mean()) < 1e-4
    assert abs(loss - (math.log(50257) + 0.0002 * 768)) < 0.15
    m.backward()
    norm = m.step(lr=6e-4)
    assert math.isfinite(norm) and norm > 0
    loss2 = m.forward(dev(x), dev(y))
    assert loss2 < loss


def test_checkpoint_resume_is_bit_exact(tmp_path):
    """Three steps in one run against two steps, a checkpoint, a fresh model
    (other seed) that loads it, and the third step: parameters, Adam moments
    and the next loss identical bit for bit (the pages' ckpt.pt resume)."""
    c = oracle_cfg(CONFIGS["char"], batch_size=2, n_layer=2)
    batches = [synthdata.markov_batch(65, c.batch_size, c.seq_len, 700 + i) for i in range(3)]

    def run(m, steps):
        loss = None
        for x, y in steps:
            m.zero_grad()
            loss = m.forward(dev(x), dev(y))
            m.backward()
            m.step(lr=2e-3)
        return loss

    for precision in (gpt2.GPT2_BF16, gpt2.GPT2_FP32):
        a = gpt2.GPT2(gpu_cfg(c, precision), seed=21)
        la = run(a, batches)
        b = gpt2.GPT2(gpu_cfg(c, precision), seed=21)
        run(b, batches[:2])
        path = tmp_path / f"ckpt{precision}.bin"
        b.save(path)
        r = gpt2.GPT2(gpu_cfg(c, precision), seed=99)
        r.load(path)
        lr_ = run(r, batches[2:])
        assert lr_ == la, (precision, lr_, la)
        for which in (gpt2.GPT2_PARAM, gpt2.GPT2_ADAM_M, gpt2.GPT2_ADAM_V):
            sa, sr = a.state(which), r.state(which)
            for n in sa:
                assert np.array_equal(sa[n], sr[n]), (precision, which, n)
        # a checkpoint of another configuration is refused
        other = gpt2.GPT2(gpu_cfg(oracle_cfg(c, n_layer=1), precision), seed=1)
        with pytest.raises(gpt2.GPT2Error):
            other.load(path)
        for m in (a, b, r, other):
            m.close()
