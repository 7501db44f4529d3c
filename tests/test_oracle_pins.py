"""Pins for the oracle: checks against what the pages and the mathematics fix,
independent of the oracle's own formulas and of the CUDA library.

Each test names the passage or the fact it rests on. A plausible mistake in
the oracle (a dropped term, a wrong sign or index, a transposed operand, a
wrong scale) fails at least one of them:
  * parameter counts (pages) pin every tensor shape;
  * initial loss ~ ln V (pages) pins the init scale and the LayerNorm;
  * causality pins the mask direction;
  * library routines (torch fp64: layer_norm, SDPA is_causal, gelu tanh,
    cross_entropy ignore_index, AdamW, clip_grad_norm_) pin each layer, and
    torch autograd on a model composed of them pins the whole backward;
  * central finite differences pin the backward against the forward;
  * closed forms: T=1 attention, q=0 prefix mean, AdamW step 1, clip;
  * the schedule values printed in the nanoGPT guide Lab 4.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import synthdata
from oracle import gpt2_oracle as O
from oracle import CONFIGS



@pytest.fixture(autouse=True)
def _fp64_default():
    """The library-routine pins below build fp64 torch tensors with default
    dtypes; the default is set for each test of this module only and restored
    afterwards, so other test modules keep torch's fp32 default."""
    old = torch.get_default_dtype()
    torch.set_default_dtype(torch.float64)
    yield
    torch.set_default_dtype(old)


def tiny(**kw):
    c = O.Config(**{**CONFIGS["tiny"].__dict__, **kw})
    return c


# ----------------------------------------------------------------------------
# shapes and counts
# ----------------------------------------------------------------------------
def test_param_counts_match_pages(page_values):
    cfg = CONFIGS["gpt2_124m"]
    excl_wpe = O.num_params(cfg, include_wpe=False)
    total = O.num_params(cfg)
    wte = cfg.vocab_size * cfg.d_model
    assert round(excl_wpe / 1e6, 2) == page_values["params_gpt2_excl_wpe_millions"]
    assert round(wte / 1e6, 1) == page_values["wte_millions"]
    assert round(100 * wte / total) == page_values["wte_fraction_percent"]
    assert round(total / 1e6) == page_values["gpt2_total_millions"]
    assert cfg.Vp == page_values["vocab_padded"] and cfg.vocab_size == page_values["vocab_gpt2"]
    # exact integers of the same counts
    assert excl_wpe == 123_653_376 and total == 124_439_808
    assert O.num_params(cfg, padded=True) == 124_475_904
    assert O.num_params(CONFIGS["tiny"]) == 108_352


def test_tokens_per_iter_arithmetic(page_values):
    assert 40 * 12 * 1024 == page_values["tokens_per_iter_gpt2"]
    assert 1 * 12 * 64 == page_values["tokens_per_iter_cpu"]


def test_vocab_rounding_default():
    assert O.Config(1, 1, 8, 65, 8, 1, 8).Vp == 128
    assert O.Config(1, 1, 8, 50257, 8, 1, 8).Vp == 50304  # 50304 = 393 * 128


# ----------------------------------------------------------------------------
# init
# ----------------------------------------------------------------------------
def test_init_normals_are_standard_normal():
    from scipy import stats
    z = O.init_normals(1337, 3, 200_000)
    assert stats.kstest(z, "norm").pvalue > 1e-3
    assert abs(z.mean()) < 5 / math.sqrt(z.size)
    assert abs(z.var() - 1) < 5 * math.sqrt(2 / z.size)
    # different tensors, different seeds -> different streams
    assert not np.array_equal(O.init_normals(1337, 3, 100), O.init_normals(1337, 4, 100))
    assert not np.array_equal(O.init_normals(1337, 3, 100), O.init_normals(1338, 3, 100))


def test_init_scales_follow_pages():
    cfg = O.Config(n_layer=12, n_head=4, d_model=128, vocab_size=1000, block_size=64,
                   batch_size=1, seq_len=8)
    p = O.init_params(cfg, 7)
    for name, a in p.items():
        if name.endswith(".g"):
            assert np.all(a == 1.0)
        elif name.endswith(".b"):
            assert np.all(a == 0.0)
        else:
            std = 0.02 / math.sqrt(2 * 12) if name.endswith("proj.W") else 0.02
            tol = 4 * std * math.sqrt(2.0 / a.size)
            assert abs(a.std() - std) < tol, name
            assert abs(a.mean()) < 4 * std / math.sqrt(a.size), name
            assert np.all(a == a.astype(np.float32).astype(np.float64))  # fp32 master


# ----------------------------------------------------------------------------
# initial loss ~ ln V
# ----------------------------------------------------------------------------
def _init_loss(cfg, seed=1, kind="uniform"):
    p = O.init_params(cfg, seed)
    x, y = synthdata.batch_for(kind, cfg.vocab_size, cfg.batch_size, cfg.seq_len, 99)
    loss, _, _ = O.forward(p, cfg, x, y)
    return loss


def test_initial_loss_is_ln_vocab_small(page_values):
    # logits ~ N(0, 0.02^2 d) at init, so E[loss] ~ ln V + 0.02^2 d / 2
    cfg = CONFIGS["tiny"]
    loss = _init_loss(cfg)
    assert abs(loss - page_values["init_loss_v65"]) < 0.1
    assert abs(loss - (math.log(65) + 0.0002 * cfg.d_model)) < 0.05


def test_initial_loss_is_ln_vocab_gpt2_width(page_values):
    cfg = O.Config(n_layer=2, n_head=12, d_model=768, vocab_size=50257, padded_vocab=50304,
                   block_size=1024, batch_size=1, seq_len=64)
    loss = _init_loss(cfg, kind="zipf")
    assert abs(math.log(50257) - page_values["init_loss_v50257"]) < 0.01
    assert abs(loss - (page_values["init_loss_v50257"] + 0.0002 * 768)) < 0.1


# ----------------------------------------------------------------------------
# causality
# ----------------------------------------------------------------------------
def test_causality_future_tokens_do_not_change_past_logits():
    cfg = CONFIGS["tiny"]
    p = O.init_params(cfg, 3)
    x, _ = synthdata.uniform_batch(65, cfg.batch_size, cfg.seq_len, 5)
    _, z0, _ = O.forward(p, cfg, x)
    t0 = 37
    x2 = x.copy()
    x2[:, t0 + 1:] = (x2[:, t0 + 1:] + 11) % 65
    _, z1, _ = O.forward(p, cfg, x2)
    assert np.array_equal(z0[:, :t0 + 1], z1[:, :t0 + 1])
    assert not np.allclose(z0[:, t0 + 1:], z1[:, t0 + 1:])


# ----------------------------------------------------------------------------
# layer-level pins against library routines
# ----------------------------------------------------------------------------
def test_layernorm_matches_torch_and_normalises():
    rng = np.random.default_rng(0)
    x = rng.normal(2.0, 3.0, (5, 7, 48))
    g, b = rng.normal(size=48), rng.normal(size=48)
    y, mu, rstd = O.layernorm_fwd(x, g, b)
    ref = F.layer_norm(torch.tensor(x), (48,), torch.tensor(g), torch.tensor(b), eps=1e-5)
    assert np.allclose(y, ref.numpy(), atol=1e-12, rtol=0)
    y1, _, _ = O.layernorm_fwd(x, np.ones(48), np.zeros(48))
    assert np.allclose(y1.mean(-1), 0, atol=1e-12)
    assert np.allclose(y1.var(-1), 1 / (1 + 1e-5 * rstd[..., 0] ** 2), atol=1e-9)


def test_layernorm_backward_matches_autograd():
    rng = np.random.default_rng(1)
    x = rng.normal(size=(6, 32)); g = rng.normal(size=32); b = rng.normal(size=32)
    dy = rng.normal(size=(6, 32))
    _, mu, rstd = O.layernorm_fwd(x, g, b)
    dx, dg, db = O.layernorm_bwd(dy, x, g, mu, rstd)
    xt, gt, bt = (torch.tensor(a, requires_grad=True) for a in (x, g, b))
    F.layer_norm(xt, (32,), gt, bt, eps=1e-5).backward(torch.tensor(dy))
    for a, t in ((dx, xt), (dg, gt), (db, bt)):
        assert np.allclose(a, t.grad.numpy(), atol=1e-11, rtol=0)


def test_gelu_is_tanh_form_not_erf(page_values):
    x = np.linspace(-6, 6, 1001)
    ref = F.gelu(torch.tensor(x), approximate="tanh").numpy()
    assert np.allclose(O.gelu_tanh(x), ref, atol=1e-14, rtol=0)
    from scipy.special import erf
    exact = 0.5 * (1 + erf(1 / math.sqrt(2)))
    diff = abs(O.gelu_tanh(np.array(1.0)) - exact)
    assert page_values["gelu_forms_differ"] == 1 and 1e-4 < diff < 2e-4
    xt = torch.tensor(x, requires_grad=True)
    F.gelu(xt, approximate="tanh").sum().backward()
    assert np.allclose(O.gelu_tanh_grad(x), xt.grad.numpy(), atol=1e-13, rtol=0)


def test_attention_matches_sdpa_causal():
    rng = np.random.default_rng(2)
    q, k, v = (rng.normal(size=(2, 3, 17, 8)) for _ in range(3))
    o = O.attention_fwd(q, k, v)
    qt, kt, vt = (torch.tensor(a, requires_grad=True) for a in (q, k, v))
    ref = F.scaled_dot_product_attention(qt, kt, vt, is_causal=True)
    assert np.allclose(o, ref.detach().numpy(), atol=1e-13, rtol=0)
    do = rng.normal(size=o.shape)
    ref.backward(torch.tensor(do))
    dq, dk, dv = O.attention_bwd(do, q, k, v)
    for a, t in ((dq, qt), (dk, kt), (dv, vt)):
        assert np.allclose(a, t.grad.numpy(), atol=1e-12, rtol=0)


def test_attention_closed_forms():
    rng = np.random.default_rng(3)
    # T = 1: the only visible key is itself, o = v
    q, k, v = (rng.normal(size=(1, 2, 1, 8)) for _ in range(3))
    assert np.allclose(O.attention_fwd(q, k, v), v, atol=0, rtol=0)
    # q = 0: uniform weights over the visible prefix, o_i = mean(v_0..v_i)
    T = 9
    k, v = rng.normal(size=(1, 1, T, 4)), rng.normal(size=(1, 1, T, 4))
    o = O.attention_fwd(np.zeros((1, 1, T, 4)), k, v)
    prefix_mean = np.cumsum(v, axis=2) / np.arange(1, T + 1)[None, None, :, None]
    assert np.allclose(o, prefix_mean, atol=1e-14)
    # lse: q = 0 gives log(i + 1); otherwise torch.logsumexp of the masked scores
    lse0 = O.causal_lse(np.zeros((1, 1, T, 4)), k)
    assert np.allclose(lse0[0, 0], np.log(np.arange(1, T + 1)), atol=1e-14)
    qq = rng.normal(size=(1, 1, T, 4))
    s = torch.tensor(qq[0, 0] @ k[0, 0].T / 2.0)
    s = s.masked_fill(torch.triu(torch.ones(T, T, dtype=torch.bool), 1), float("-inf"))
    assert np.allclose(O.causal_lse(qq, k)[0, 0], torch.logsumexp(s, -1).numpy(), atol=1e-13)
    # rows of P sum to one and are zero above the diagonal
    P = O.causal_softmax(rng.normal(size=(1, 1, T, 4)), k)
    assert np.allclose(P.sum(-1), 1.0, atol=1e-14)
    assert np.all(np.triu(P[0, 0], 1) == 0.0)


# ----------------------------------------------------------------------------
# the whole model against torch autograd over library routines
# ----------------------------------------------------------------------------
def _torch_model_loss(params, cfg, x, y):
    """Same architecture composed of torch library routines (fp64)."""
    P = {n: torch.tensor(a, requires_grad=True) for n, a in params.items()}
    B, T = x.shape
    xi = torch.tensor(x, dtype=torch.long)
    h = F.embedding(xi, P["wte"]) + P["wpe"][:T]
    H, hs, C = cfg.n_head, cfg.hs, cfg.d_model
    for l in range(cfg.n_layer):
        g = lambda n: P[f"h{l}.{n}"]
        u = F.layer_norm(h, (C,), g("ln1.g"), g("ln1.b"), eps=1e-5)
        q, k, v = F.linear(u, g("attn.W"), g("attn.b")).split(C, dim=2)
        q, k, v = (t.view(B, T, H, hs).transpose(1, 2) for t in (q, k, v))
        o = F.scaled_dot_product_attention(q, k, v, is_causal=True).transpose(1, 2).reshape(B, T, C)
        h = h + F.linear(o, g("attn_proj.W"), g("attn_proj.b"))
        u2 = F.layer_norm(h, (C,), g("ln2.g"), g("ln2.b"), eps=1e-5)
        h = h + F.linear(F.gelu(F.linear(u2, g("fc.W"), g("fc.b")), approximate="tanh"),
                         g("mlp_proj.W"), g("mlp_proj.b"))
    uf = F.layer_norm(h, (C,), P["lnf.g"], P["lnf.b"], eps=1e-5)
    logits = F.linear(uf, P["wte"][:cfg.vocab_size])
    loss = F.cross_entropy(logits.view(-1, cfg.vocab_size), torch.tensor(y, dtype=torch.long).view(-1),
                           ignore_index=-1)
    return loss, logits, P


def test_model_forward_backward_match_torch_autograd():
    cfg = CONFIGS["tiny"]
    params = O.init_params(cfg, 11)
    # non-trivial LN/bias values so that every term is exercised
    rng = np.random.default_rng(4)
    for n in params:
        if n.endswith(".g") or n.endswith(".b"):
            params[n] = params[n] + 0.1 * rng.normal(size=params[n].shape)
    x, y = synthdata.uniform_batch(65, cfg.batch_size, cfg.seq_len, 12)
    y = y.copy()
    y[1, 5] = -1
    y[3, :7] = -1  # ignore_index rows
    loss, logits, cache = O.forward(params, cfg, x, y)
    grads = O.backward(params, cfg, cache)
    tl, tlogits, P = _torch_model_loss(params, cfg, x, y)
    tl.backward()
    assert abs(loss - tl.item()) < 1e-13
    assert np.allclose(logits, tlogits.detach().numpy(), atol=1e-12, rtol=0)
    for n, g in grads.items():
        ref = P[n].grad.numpy()
        err = np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-300)
        assert err < 1e-10, (n, err)
    assert np.all(grads["wte"][cfg.vocab_size:] == 0.0)  # pad rows get nothing


def test_finite_differences_tiny():
    cfg = CONFIGS["tiny"]
    params = O.init_params(cfg, 21)
    x, y = synthdata.uniform_batch(65, cfg.batch_size, cfg.seq_len, 22)
    _, _, cache = O.forward(params, cfg, x, y)
    grads = O.backward(params, cfg, cache)
    rng = np.random.default_rng(5)
    h = 1e-5
    checked = 0
    for name, shape in O.param_shapes(cfg):
        n = int(np.prod(shape))
        rows = cfg.vocab_size if name == "wte" else shape[0]
        hi = rows * (shape[1] if len(shape) == 2 else 1)
        for idx in rng.choice(hi, size=min(8, hi), replace=False):
            flat = params[name].reshape(-1)
            old = flat[idx]
            flat[idx] = old + h
            lp, _, _ = O.forward(params, cfg, x, y)
            flat[idx] = old - h
            lm, _, _ = O.forward(params, cfg, x, y)
            flat[idx] = old
            fd = (lp - lm) / (2 * h)
            an = grads[name].reshape(-1)[idx]
            assert abs(fd - an) <= 1e-6 * abs(an) + 2e-10, (name, idx, fd, an)
            checked += 1
    assert checked >= 200


def test_cross_entropy_gradient_rows_sum_to_zero():
    cfg = CONFIGS["tiny"]
    params = O.init_params(cfg, 2)
    x, y = synthdata.uniform_batch(65, cfg.batch_size, cfg.seq_len, 3)
    _, _, cache = O.forward(params, cfg, x, y)
    O.backward(params, cfg, cache)
    assert np.allclose(cache["dz"].sum(-1), 0.0, atol=1e-15)


def test_grad_accumulation_equivalence():
    """1 x B equals 4 x B/4 with the loss divided by the micro-batch count
    (sotaaz Section 3; nanoGPT guide Lab 5)."""
    base = CONFIGS["tiny"]
    params = O.init_params(base, 31)
    x, y = synthdata.uniform_batch(65, 8, base.seq_len, 32)
    c1 = O.Config(**{**base.__dict__, "batch_size": 8})
    _, _, cache = O.forward(params, c1, x, y)
    g1 = O.backward(params, c1, cache)
    c4 = O.Config(**{**base.__dict__, "batch_size": 2, "grad_accum_steps": 4})
    g4 = O.zero_grads(params)
    for i in range(4):
        _, _, cache = O.forward(params, c4, x[2 * i:2 * i + 2], y[2 * i:2 * i + 2])
        O.backward(params, c4, cache, g4)
    for n in g1:
        err = np.linalg.norm(g1[n] - g4[n]) / max(np.linalg.norm(g1[n]), 1e-300)
        assert err < 1e-12, (n, err)


# ----------------------------------------------------------------------------
# optimizer pins
# ----------------------------------------------------------------------------
def test_clip_matches_torch_and_caps_norm():
    rng = np.random.default_rng(6)
    for scale in (0.01, 10.0):
        grads = {"a": scale * rng.normal(size=(7, 3)), "b": scale * rng.normal(size=11)}
        tg = [torch.tensor(g) for g in grads.values()]
        ts = [torch.zeros_like(t, requires_grad=True) for t in tg]
        for t, g in zip(ts, tg):
            t.grad = g.clone()
        tn = torch.nn.utils.clip_grad_norm_(ts, 1.0).item()
        n = O.clip_grads(grads, 1.0)
        assert abs(n - tn) < 1e-12 * max(1, tn)
        for g, t in zip(grads.values(), ts):
            assert np.allclose(g, t.grad.numpy(), atol=1e-15, rtol=1e-14)
        assert abs(O.global_grad_norm(grads) - min(n, 1.0)) < 1e-6


def test_adamw_matches_torch_over_steps():
    rng = np.random.default_rng(7)
    W = rng.normal(size=(5, 4)); b = rng.normal(size=4)
    tW, tb = torch.tensor(W, requires_grad=True), torch.tensor(b, requires_grad=True)
    opt = torch.optim.AdamW([{"params": [tW], "weight_decay": 0.1},
                             {"params": [tb], "weight_decay": 0.0}],
                            lr=1e-3, betas=(0.9, 0.95), eps=1e-8)
    mW, vW, mb, vb = (np.zeros_like(a) for a in (W, W, b, b))
    for t in range(1, 6):
        gW, gb = rng.normal(size=W.shape), rng.normal(size=b.shape)
        tW.grad, tb.grad = torch.tensor(gW), torch.tensor(gb)
        opt.step()
        O.adamw_update(W, gW, mW, vW, t, 1e-3, 0.9, 0.95, 1e-8, 0.1, decay=True)
        O.adamw_update(b, gb, mb, vb, t, 1e-3, 0.9, 0.95, 1e-8, 0.1, decay=False)
        assert np.allclose(W, tW.detach().numpy(), atol=1e-15, rtol=1e-13)
        assert np.allclose(b, tb.detach().numpy(), atol=1e-15, rtol=1e-13)


def _torch_gpt_modules(cfg):
    """The model's parameters held by real torch modules (nn.Embedding,
    nn.Linear, nn.LayerNorm; the LM head is the token embedding, tied), keyed
    by the oracle's names. Shapes come from the modules, not from the oracle."""
    C, L = cfg.d_model, cfg.n_layer
    mods = torch.nn.ModuleDict({"wte": torch.nn.Embedding(cfg.Vp, C),
                                "wpe": torch.nn.Embedding(cfg.block_size, C)})
    for l in range(L):
        mods[f"h{l}_ln1"] = torch.nn.LayerNorm(C)
        mods[f"h{l}_attn"] = torch.nn.Linear(C, 3 * C)
        mods[f"h{l}_attn_proj"] = torch.nn.Linear(C, C)
        mods[f"h{l}_ln2"] = torch.nn.LayerNorm(C)
        mods[f"h{l}_fc"] = torch.nn.Linear(C, 4 * C)
        mods[f"h{l}_mlp_proj"] = torch.nn.Linear(4 * C, C)
    mods["lnf"] = torch.nn.LayerNorm(C)
    named = {"wte": mods["wte"].weight, "wpe": mods["wpe"].weight,
             "lnf.g": mods["lnf"].weight, "lnf.b": mods["lnf"].bias}
    for l in range(L):
        for part in ("ln1", "ln2"):
            named[f"h{l}.{part}.g"] = mods[f"h{l}_{part}"].weight
            named[f"h{l}.{part}.b"] = mods[f"h{l}_{part}"].bias
        for part in ("attn", "attn_proj", "fc", "mlp_proj"):
            named[f"h{l}.{part}.W"] = mods[f"h{l}_{part}"].weight
            named[f"h{l}.{part}.b"] = mods[f"h{l}_{part}"].bias
    return named


def test_decay_groups_follow_configure_optimizers():
    """Which tensors weight decay touches (nanoGPT guide, Deep dive 1
    configure_optimizers: parameters of two or more dimensions decay, i.e. the
    embeddings and every Linear weight; biases and LayerNorm gains/shifts do
    not; sotaaz Section 3: decay on 2-D params only). Two pins:
    (1) by category, as the pages list them: the oracle decays exactly wte,
    wpe and the four Linear weights of each block;
    (2) by the library optimizer: two clipped steps of torch AdamW with the
    parameter groups built the pages' way over real torch modules match the
    oracle's Trainer.step on the same gradients. Decaying a 1-D tensor, or
    sparing wpe, fails both."""
    cfg = CONFIGS["tiny"]
    shapes = dict(O.param_shapes(cfg))
    decayed = {n for n, s in shapes.items() if O.decays(n, s)}
    linear_w = {f"h{l}.{p}.W" for l in range(cfg.n_layer)
                for p in ("attn", "attn_proj", "fc", "mlp_proj")}
    assert decayed == {"wte", "wpe"} | linear_w

    named = _torch_gpt_modules(cfg)
    assert set(named) == set(shapes)
    for n, p in named.items():
        assert tuple(p.shape) == tuple(shapes[n]), n
    tr = O.Trainer(cfg, 5)
    with torch.no_grad():
        for n, p in named.items():
            p.copy_(torch.tensor(tr.params[n]))
    groups = [{"params": [p for p in named.values() if p.dim() >= 2], "weight_decay": 0.1},
              {"params": [p for p in named.values() if p.dim() < 2], "weight_decay": 0.0}]
    opt = torch.optim.AdamW(groups, lr=3e-3, betas=(0.9, 0.95), eps=1e-8)
    for step in range(2):
        x, y = synthdata.uniform_batch(65, cfg.batch_size, cfg.seq_len, 40 + step)
        tr.zero_grad()
        tr.forward(x, y)
        tr.backward()
        for n, p in named.items():
            p.grad = torch.tensor(tr.grads[n]).clone()
        tn = torch.nn.utils.clip_grad_norm_(list(named.values()), 1.0).item()
        opt.step()
        n_orc = tr.step(lr=3e-3, weight_decay=0.1, clip=1.0)
        assert abs(n_orc - tn) <= 1e-12 * tn
        for n, p in named.items():
            d = float(np.abs(tr.params[n] - p.detach().numpy()).max())
            assert d < 1e-14, (step, n, d)


def test_adamw_first_step_closed_form():
    rng = np.random.default_rng(8)
    p0 = rng.normal(size=100); g = rng.normal(size=100)
    p = p0.copy(); m = np.zeros(100); v = np.zeros(100)
    lr, wd, eps = 1e-3, 0.1, 1e-8
    O.adamw_update(p, g, m, v, 1, lr, 0.9, 0.95, eps, wd, decay=True)
    assert np.allclose(p, p0 * (1 - lr * wd) - lr * g / (np.abs(g) + eps), atol=1e-15)


def test_schedule_values_from_lab4(page_values):
    pv = page_values
    W, Hz, mx, mn = int(pv["sched_warmup"]), int(pv["sched_horizon"]), pv["sched_lr_max"], pv["sched_lr_min"]
    f = lambda it: O.lr_schedule(it, W, Hz, mx, mn)
    assert abs(f(0) - pv["sched_lr_at_0"]) < 1e-12
    assert abs(f(2000) - pv["sched_lr_at_2000"]) < 1e-12
    assert abs(f(301000) - pv["sched_lr_at_301000"]) < 1e-12
    assert abs(f(700000) - pv["sched_lr_at_700000"]) < 1e-12
    assert abs(f(600000) - mn) < 1e-12 and f(1000) < f(1998) < f(1999) == f(2000)
    # the 124M recipe: 715 warmup steps (sotaaz Section 3)
    assert abs(O.lr_schedule(0, 715, 19073, 6e-4, 6e-5) - 6e-4 / 715) < 1e-15


# ----------------------------------------------------------------------------
# end to end: overfitting one batch
# ----------------------------------------------------------------------------
@pytest.mark.slow
def test_overfit_single_batch():
    """Loss on one fixed batch falls toward zero ("Let's reproduce GPT-2"
    00:56:42: overfit a single batch)."""
    cfg = CONFIGS["tiny"]
    tr = O.Trainer(cfg, 1337)
    x, y = synthdata.uniform_batch(65, cfg.batch_size, cfg.seq_len, 1337)
    first = None
    for it in range(300):
        tr.zero_grad()
        loss, _ = tr.forward(x, y)
        first = loss if first is None else first
        tr.backward()
        tr.step(lr=1e-3 if it < 250 else 5e-4, weight_decay=0.0)
    loss, _ = tr.forward(x, y)
    assert loss < 0.1 * first
