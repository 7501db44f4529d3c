"""Plain CPU oracle for one GPT-2 training iteration (fp64 numpy).

TEST INFRASTRUCTURE ONLY. This module is the checker that the CUDA library is
compared against. Only the test suite, the smoke check and the benchmark's CPU
baseline may import it; the library never calls it and shares no code with it.

What it computes follows the pages:
  * "Let's reproduce GPT-2 (124M)" (library.recl.app summary): Core
    Architecture; 01:06:14 weight tying; 01:13:47 init std 0.02 with residual
    init; 02:06:54 vocab 50257 -> 50304; 02:21:06 warmup + cosine.
  * "Andrej Karpathy: Let's reproduce GPT-2" (youtube.nixfred.com): "Writing
    the network so it matches the real thing" (tying, init 1/sqrt(2L)).
  * "Karpathy's Let's Reproduce GPT-2 in One Read" (sotaaz.com): "One check we
    ran: the GELU" (tanh approximation); Section 3 (AdamW betas/eps, clip 1.0,
    warmup/cosine, decay on 2-D params only, dividing each micro-batch loss by
    the number of micro-batches).
  * "nanoGPT" guide (stanleyjacob.dev): Part IV Stages 1-5 (schedule, the
    micro-step loop, cross_entropy with ignore_index=-1, clip then step);
    Deep dive 1 (attention shape choreography, manual attention semantics,
    init, decay-by-rank, tied parameter counting).
  * "Build GPT from scratch" (byteknotlabs): "The model in forty lines"
    (pre-norm block, nn.LayerNorm, mask with -inf before softmax).

Readings where the pages are silent (each also listed in the design notes):
  LayerNorm eps = 1e-5 (nn.LayerNorm default), biased variance; GELU tanh
  constants from Hendrycks & Gimpel; pad vocabulary columns masked out of the
  softmax; block_size = T; clip with PyTorch clip_grad_norm_ semantics
  (coef = min(1, clip/(norm + 1e-6))); AdamW in the PyTorch form (decoupled
  decay p *= 1 - lr*wd first, bias-corrected moments, eps outside the sqrt);
  init from SplitMix64 + Box-Muller as specified in ``init_params``.

Nothing here is blocked, fused or reordered beyond the definitions: matmuls
are numpy matmuls of whole tensors.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

LN_EPS = 1e-5
CLIP_EPS = 1e-6


# ----------------------------------------------------------------------------
# configuration
# ----------------------------------------------------------------------------
@dataclass
class Config:
    n_layer: int
    n_head: int
    d_model: int
    vocab_size: int
    block_size: int
    batch_size: int
    seq_len: int
    padded_vocab: int = 0          # 0 -> round vocab_size up to a multiple of 128
    grad_accum_steps: int = 1

    @property
    def Vp(self) -> int:
        if self.padded_vocab:
            return self.padded_vocab
        return ((self.vocab_size + 127) // 128) * 128

    @property
    def hs(self) -> int:
        return self.d_model // self.n_head


# ----------------------------------------------------------------------------
# parameters: canonical order and init
# ----------------------------------------------------------------------------
def param_shapes(cfg: Config):
    """Canonical parameter list (nanoGPT guide, Deep dive 1; GPT-2 uses biases).

    wte [Vp, d] is the token embedding and, tied, the LM head
    ("Let's reproduce GPT-2", 01:06:14). Linear weights are [out, in].
    """
    d, L = cfg.d_model, cfg.n_layer
    out = [("wte", (cfg.Vp, d)), ("wpe", (cfg.block_size, d))]
    for l in range(L):
        p = f"h{l}."
        out += [
            (p + "ln1.g", (d,)), (p + "ln1.b", (d,)),
            (p + "attn.W", (3 * d, d)), (p + "attn.b", (3 * d,)),
            (p + "attn_proj.W", (d, d)), (p + "attn_proj.b", (d,)),
            (p + "ln2.g", (d,)), (p + "ln2.b", (d,)),
            (p + "fc.W", (4 * d, d)), (p + "fc.b", (4 * d,)),
            (p + "mlp_proj.W", (d, 4 * d)), (p + "mlp_proj.b", (d,)),
        ]
    out += [("lnf.g", (d,)), ("lnf.b", (d,))]
    return out


def decays(name: str, shape) -> bool:
    """Weight decay only on parameters with two or more dimensions
    (nanoGPT guide, Deep dive 1 configure_optimizers; sotaaz Section 3)."""
    return len(shape) >= 2


def num_params(cfg: Config, include_wpe: bool = True, padded: bool = False) -> int:
    """Parameter count with the tied matrix counted once (nanoGPT guide,
    Deep dive 1, "the famous trap in this file is parameter counting")."""
    n = 0
    for name, shape in param_shapes(cfg):
        if name == "wpe" and not include_wpe:
            continue
        if name == "wte" and not padded:
            shape = (cfg.vocab_size, shape[1])
        n += int(np.prod(shape))
    return n


_GAMMA = 0x9E3779B97F4A7C15
_MASK = (1 << 64) - 1


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
    return z ^ (z >> np.uint64(31))


def init_normals(seed: int, k: int, n: int) -> np.ndarray:
    """Standard normals for element i = 0..n-1 of tensor number k.

    Specification (the pages fix only the law N(0, 0.02^2)): start a
    SplitMix64 generator at state = seed XOR (k * 2^40 + i); its first two
    outputs r1, r2 give u1 = (r1 >> 11 + 1) * 2^-53 in (0, 1] and
    u2 = (r2 >> 11) * 2^-53 in [0, 1); z = sqrt(-2 ln u1) cos(2 pi u2)
    (Box & Muller 1958), in double precision.
    """
    with np.errstate(over="ignore"):
        i = np.arange(n, dtype=np.uint64)
        state = np.uint64(seed & _MASK) ^ (np.uint64(k) * np.uint64(1 << 40) + i)
        r1 = _mix64(state + np.uint64(_GAMMA))
        r2 = _mix64(state + np.uint64((2 * _GAMMA) & _MASK))
    u1 = ((r1 >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
    u2 = (r2 >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)


def init_params(cfg: Config, seed: int):
    """GPT-2 init ("Let's reproduce GPT-2" 01:13:47; nixfred "Initialization";
    nanoGPT guide Deep dive 1): every matrix and both embeddings N(0, 0.02^2);
    the two projections that write into the residual stream (attn_proj.W,
    mlp_proj.W) N(0, (0.02/sqrt(2 n_layer))^2); biases 0; LayerNorm gain 1,
    shift 0. Values are rounded to fp32, the precision the master copy keeps
    (nixfred "Precision": parameters stay in higher precision), then held in
    fp64 here. Pad rows wte[V:Vp] are initialised like the rest."""
    params = {}
    resid_std = 0.02 / math.sqrt(2 * cfg.n_layer)
    for k, (name, shape) in enumerate(param_shapes(cfg)):
        n = int(np.prod(shape))
        if name.endswith(".g"):
            v = np.ones(n)
        elif name.endswith(".b"):
            v = np.zeros(n)
        else:
            std = resid_std if (name.endswith("attn_proj.W") or name.endswith("mlp_proj.W")) else 0.02
            v = (std * init_normals(seed, k, n)).astype(np.float32).astype(np.float64)
        params[name] = v.reshape(shape)
    return params


# ----------------------------------------------------------------------------
# layer definitions
# ----------------------------------------------------------------------------
def layernorm_fwd(x, g, b, eps=LN_EPS):
    """Per-row LayerNorm with affine gain/shift (nn.LayerNorm semantics,
    byteknotlabs "The model in forty lines"; biased variance)."""
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    rstd = 1.0 / np.sqrt(var + eps)
    xhat = (x - mu) * rstd
    return xhat * g + b, mu, rstd


def layernorm_bwd(dy, x, g, mu, rstd):
    """Analytic gradient of layernorm_fwd: dxhat = dy*g,
    dx = rstd * (dxhat - mean(dxhat) - xhat * mean(dxhat * xhat))."""
    xhat = (x - mu) * rstd
    dxhat = dy * g
    dx = rstd * (dxhat - dxhat.mean(axis=-1, keepdims=True)
                 - xhat * (dxhat * xhat).mean(axis=-1, keepdims=True))
    dg = (dy * xhat).reshape(-1, x.shape[-1]).sum(axis=0)
    db = dy.reshape(-1, x.shape[-1]).sum(axis=0)
    return dx, dg, db


_GELU_A = math.sqrt(2.0 / math.pi)
_GELU_C = 0.044715


def gelu_tanh(x):
    """GPT-2's GELU, the tanh approximation (sotaaz "One check we ran: the
    GELU in nanoGPT is not GPT-2's"): 0.5 x (1 + tanh(sqrt(2/pi)(x + 0.044715 x^3)))
    (Hendrycks & Gimpel 2016)."""
    return 0.5 * x * (1.0 + np.tanh(_GELU_A * (x + _GELU_C * x ** 3)))


def gelu_tanh_grad(x):
    """d/dx of gelu_tanh."""
    t = np.tanh(_GELU_A * (x + _GELU_C * x ** 3))
    return 0.5 * (1.0 + t) + 0.5 * x * (1.0 - t * t) * _GELU_A * (1.0 + 3.0 * _GELU_C * x * x)


def causal_softmax(q, k):
    """P = softmax(q k^T / sqrt(hs)) with positions j > i set to -inf before
    the softmax (nanoGPT guide Deep dive 1, the manual path; byteknotlabs
    "Common pitfalls": mask before softmax, -inf not 0). q, k: [..., T, hs]."""
    T, hs = q.shape[-2], q.shape[-1]
    s = (q @ np.swapaxes(k, -1, -2)) / math.sqrt(hs)
    future = np.triu(np.ones((T, T), dtype=bool), k=1)
    s = np.where(future, -np.inf, s)
    s = s - s.max(axis=-1, keepdims=True)
    e = np.exp(s)
    return e / e.sum(axis=-1, keepdims=True)


def causal_lse(q, k):
    """Natural-log normaliser of each causal softmax row,
    lse_i = log sum_{j<=i} exp(q_i . k_j / sqrt(hs)); flash-style kernels keep
    it from the forward to rebuild P in the backward."""
    T, hs = q.shape[-2], q.shape[-1]
    s = (q @ np.swapaxes(k, -1, -2)) / math.sqrt(hs)
    future = np.triu(np.ones((T, T), dtype=bool), k=1)
    s = np.where(future, -np.inf, s)
    mx = s.max(axis=-1, keepdims=True)
    return (mx + np.log(np.exp(s - mx).sum(axis=-1, keepdims=True)))[..., 0]


def attention_fwd(q, k, v):
    """o = P v for P = causal_softmax(q, k). Shapes [B, H, T, hs]."""
    return causal_softmax(q, k) @ v


def attention_bwd(do, q, k, v):
    """Gradient of attention_fwd. With P from the same definition:
    dV = P^T dO, dP = dO V^T, dS = P * (dP - rowsum(dP * P)),
    dQ = dS K / sqrt(hs), dK = dS^T Q / sqrt(hs)."""
    hs = q.shape[-1]
    P = causal_softmax(q, k)
    dv = np.swapaxes(P, -1, -2) @ do
    dP = do @ np.swapaxes(v, -1, -2)
    dS = P * (dP - (dP * P).sum(axis=-1, keepdims=True))
    dq = dS @ k / math.sqrt(hs)
    dk = np.swapaxes(dS, -1, -2) @ q / math.sqrt(hs)
    return dq, dk, dv


def linear(x, W, b=None):
    """PyTorch Linear: y = x W^T + b with W stored [out, in]."""
    y = x @ W.T
    return y if b is None else y + b


def split_heads(qkv, cfg: Config):
    """(B,T,3C) -> q,k,v each (B,nh,T,hs): columns [0,C) are q, [C,2C) k,
    [2C,3C) v; head h is columns h*hs..(h+1)*hs-1 of each (nanoGPT guide,
    Deep dive 1 shape choreography)."""
    B, T, _ = qkv.shape
    C, H, hs = cfg.d_model, cfg.n_head, cfg.hs
    q, k, v = qkv[..., :C], qkv[..., C:2 * C], qkv[..., 2 * C:]
    f = lambda t: t.reshape(B, T, H, hs).transpose(0, 2, 1, 3)
    return f(q), f(k), f(v)


def merge_heads(t):
    """(B,nh,T,hs) -> (B,T,C): heads side by side in order."""
    B, H, T, hs = t.shape
    return t.transpose(0, 2, 1, 3).reshape(B, T, H * hs)


# ----------------------------------------------------------------------------
# model forward / backward
# ----------------------------------------------------------------------------
def forward(params, cfg: Config, tokens, targets=None):
    """One forward pass (nanoGPT guide Part IV Stage 4; "Let's reproduce
    GPT-2" 00:31:00 and Core Architecture).

    x = wte[idx] + wpe[arange(T)]; for each block x = x + attn(ln_1(x)),
    x = x + mlp(ln_2(x)); logits = ln_f(x) wte[:V]^T (tied head, no bias;
    pad columns V..Vp-1 are masked, i.e. not part of the softmax);
    loss = mean over targets != -1 of (logsumexp(z) - z[y]).

    Returns (loss or None, logits [B,T,V], cache for backward).
    """
    tokens = np.asarray(tokens)
    B, T = tokens.shape
    V = cfg.vocab_size
    assert T <= cfg.block_size
    cache = {"tokens": tokens, "layers": []}
    x = params["wte"][tokens] + params["wpe"][:T][None, :, :]
    for l in range(cfg.n_layer):
        p = lambda n: params[f"h{l}.{n}"]
        c = {"x_in": x}
        u, c["mu1"], c["rstd1"] = layernorm_fwd(x, p("ln1.g"), p("ln1.b"))
        c["u1"] = u
        qkv = linear(u, p("attn.W"), p("attn.b"))
        q, k, v = split_heads(qkv, cfg)
        c["q"], c["k"], c["v"] = q, k, v
        o = merge_heads(attention_fwd(q, k, v))
        c["o"] = o
        x = x + linear(o, p("attn_proj.W"), p("attn_proj.b"))
        c["x_mid"] = x
        u2, c["mu2"], c["rstd2"] = layernorm_fwd(x, p("ln2.g"), p("ln2.b"))
        c["u2"] = u2
        hpre = linear(u2, p("fc.W"), p("fc.b"))
        c["hpre"] = hpre
        h = gelu_tanh(hpre)
        c["h"] = h
        x = x + linear(h, p("mlp_proj.W"), p("mlp_proj.b"))
        cache["layers"].append(c)
    cache["x_final"] = x
    uf, cache["muf"], cache["rstdf"] = layernorm_fwd(x, params["lnf.g"], params["lnf.b"])
    cache["uf"] = uf
    logits = uf @ params["wte"][:V].T
    cache["logits"] = logits
    if targets is None:
        return None, logits, cache
    targets = np.asarray(targets)
    cache["targets"] = targets
    zmax = logits.max(axis=-1, keepdims=True)
    lse = (zmax + np.log(np.exp(logits - zmax).sum(axis=-1, keepdims=True)))[..., 0]
    valid = targets != -1
    n_valid = int(valid.sum())
    zy = np.take_along_axis(logits, np.where(valid, targets, 0)[..., None], axis=-1)[..., 0]
    row_loss = np.where(valid, lse - zy, 0.0)
    cache["lse"], cache["row_loss"], cache["n_valid"] = lse, row_loss, n_valid
    loss = row_loss.sum() / max(n_valid, 1)
    return loss, logits, cache


def zero_grads(params):
    return {n: np.zeros_like(a) for n, a in params.items()}


def backward(params, cfg: Config, cache, grads=None):
    """Gradient of loss / grad_accum_steps, added (+=) into ``grads``.

    Each micro-batch loss is divided by the number of micro-batches and the
    gradients sum across backward calls ("sotaaz" Section 3; nanoGPT guide
    Deep dive 2 gradient accumulation). dz = (softmax(z) - onehot(y)) /
    (N_valid * accum) over the real vocabulary, 0 on ignored rows; pad rows
    of wte receive no gradient. Through the tie, wte gets dz^T uf plus the
    scatter of the embedding-input gradient by token; wpe[t] gets the sum over
    the batch of the same gradient at position t.
    """
    if grads is None:
        grads = zero_grads(params)
    tokens, targets = cache["tokens"], cache["targets"]
    B, T = tokens.shape
    V, d = cfg.vocab_size, cfg.d_model
    logits = cache["logits"]
    valid = targets != -1
    scale = 1.0 / (max(cache["n_valid"], 1) * cfg.grad_accum_steps)
    prob = np.exp(logits - cache["lse"][..., None])
    onehot = np.zeros_like(logits)
    np.put_along_axis(onehot, np.where(valid, targets, 0)[..., None], 1.0, axis=-1)
    dz = np.where(valid[..., None], (prob - onehot) * scale, 0.0)
    cache["dz"] = dz

    uf = cache["uf"]
    wteV = params["wte"][:V]
    grads["wte"][:V] += dz.reshape(-1, V).T @ uf.reshape(-1, d)
    duf = dz @ wteV
    dx, dg, db = layernorm_bwd(duf, cache["x_final"], params["lnf.g"], cache["muf"], cache["rstdf"])
    grads["lnf.g"] += dg
    grads["lnf.b"] += db

    for l in reversed(range(cfg.n_layer)):
        c = cache["layers"][l]
        p = lambda n: params[f"h{l}.{n}"]
        gname = lambda n: f"h{l}.{n}"
        # x_out = x_mid + h W_mp^T + b_mp
        dflat = dx.reshape(-1, d)
        grads[gname("mlp_proj.W")] += dflat.T @ c["h"].reshape(-1, 4 * d)
        grads[gname("mlp_proj.b")] += dflat.sum(axis=0)
        dh = dx @ p("mlp_proj.W")
        dhpre = dh * gelu_tanh_grad(c["hpre"])
        dhflat = dhpre.reshape(-1, 4 * d)
        grads[gname("fc.W")] += dhflat.T @ c["u2"].reshape(-1, d)
        grads[gname("fc.b")] += dhflat.sum(axis=0)
        du2 = dhpre @ p("fc.W")
        ddx, dg, db = layernorm_bwd(du2, c["x_mid"], p("ln2.g"), c["mu2"], c["rstd2"])
        grads[gname("ln2.g")] += dg
        grads[gname("ln2.b")] += db
        dx = dx + ddx
        # x_mid = x_in + o W_ap^T + b_ap
        dflat = dx.reshape(-1, d)
        grads[gname("attn_proj.W")] += dflat.T @ c["o"].reshape(-1, d)
        grads[gname("attn_proj.b")] += dflat.sum(axis=0)
        do = dx @ p("attn_proj.W")
        H, hs = cfg.n_head, cfg.hs
        do_h = do.reshape(B, T, H, hs).transpose(0, 2, 1, 3)
        dq, dk, dv = attention_bwd(do_h, c["q"], c["k"], c["v"])
        dqkv = np.concatenate([merge_heads(dq), merge_heads(dk), merge_heads(dv)], axis=-1)
        dqflat = dqkv.reshape(-1, 3 * d)
        grads[gname("attn.W")] += dqflat.T @ c["u1"].reshape(-1, d)
        grads[gname("attn.b")] += dqflat.sum(axis=0)
        du1 = dqkv @ p("attn.W")
        ddx, dg, db = layernorm_bwd(du1, c["x_in"], p("ln1.g"), c["mu1"], c["rstd1"])
        grads[gname("ln1.g")] += dg
        grads[gname("ln1.b")] += db
        dx = dx + ddx

    np.add.at(grads["wte"], tokens.reshape(-1), dx.reshape(-1, d))
    grads["wpe"][:T] += dx.sum(axis=0)
    return grads


# ----------------------------------------------------------------------------
# optimizer
# ----------------------------------------------------------------------------
def global_grad_norm(grads) -> float:
    """L2 norm over every gradient element, the tied matrix once."""
    return math.sqrt(sum(float((g * g).sum()) for g in grads.values()))


def clip_grads(grads, clip: float):
    """Clip the global norm to ``clip`` ("sotaaz" Section 3; nanoGPT guide
    Part IV Stage 5). PyTorch clip_grad_norm_ reading: every gradient is
    multiplied by min(1, clip / (norm + 1e-6)); returns the pre-clip norm."""
    n = global_grad_norm(grads)
    coef = min(1.0, clip / (n + CLIP_EPS))
    for g in grads.values():
        g *= coef
    return n


def adamw_update(p, g, m, v, t, lr, beta1, beta2, eps, wd, decay: bool):
    """One AdamW update in place (Loshchilov & Hutter, decoupled decay; the
    pages' betas (0.9, 0.95), eps 1e-8, wd 0.1 on 2-D params only, "sotaaz"
    Section 3). PyTorch form: p *= 1 - lr*wd (decayed params only);
    m = b1 m + (1-b1) g; v = b2 v + (1-b2) g^2;
    p -= lr * (m / (1-b1^t)) / (sqrt(v / (1-b2^t)) + eps)."""
    if decay:
        p *= (1.0 - lr * wd)
    m *= beta1
    m += (1.0 - beta1) * g
    v *= beta2
    v += (1.0 - beta2) * g * g
    mhat = m / (1.0 - beta1 ** t)
    vhat = v / (1.0 - beta2 ** t)
    p -= lr * mhat / (np.sqrt(vhat) + eps)


def lr_schedule(it: int, warmup: int, horizon: int, lr_max: float, lr_min: float) -> float:
    """Linear warmup then cosine decay to lr_min, then the floor
    (nanoGPT guide Part IV Stage 1 and Lab 4; "Let's reproduce GPT-2" 02:21:06).
    it < warmup: lr_max*(it+1)/warmup; it > horizon: lr_min; otherwise
    lr_min + 0.5*(1 + cos(pi*(it-warmup)/(horizon-warmup)))*(lr_max-lr_min)."""
    if it < warmup:
        return lr_max * (it + 1) / warmup
    if it > horizon:
        return lr_min
    ratio = (it - warmup) / (horizon - warmup)
    return lr_min + 0.5 * (1.0 + math.cos(math.pi * ratio)) * (lr_max - lr_min)


# ----------------------------------------------------------------------------
# generation: one sampling step
# ----------------------------------------------------------------------------
def sample_tokens(logits, temperature, top_k, u):
    """One token per row of last-position logits [B, V] ("Let's reproduce
    GPT-2" 00:37:02 the sampling loop; nanoGPT guide, sample.py): z = logits /
    temperature; with 0 < top_k < V, entries below the k-th largest z become
    -inf (the pages' topk mask keeps ties with the k-th value); p = softmax(z);
    the token is the smallest j whose cumulative p exceeds the uniform u[row]
    (inverse CDF). temperature <= 0 takes the argmax (lowest index on ties).
    Returns int64 [B]."""
    z = np.asarray(logits, dtype=np.float64)
    if temperature <= 0:
        return z.argmax(axis=1).astype(np.int64)
    z = z / temperature
    V = z.shape[1]
    if top_k is not None and 0 < top_k < V:
        kth = np.sort(z, axis=1)[:, V - top_k][:, None]
        z = np.where(z < kth, -np.inf, z)
    w = np.exp(z - z.max(axis=1, keepdims=True))
    c = np.cumsum(w, axis=1)
    target = np.asarray(u, dtype=np.float64) * c[:, -1]
    j = (c <= target[:, None]).sum(axis=1)
    last = V - 1 - np.argmax(w[:, ::-1] > 0, axis=1)
    return np.where(j >= V, last, j).astype(np.int64)


# ----------------------------------------------------------------------------
# a training-state object mirroring the library's calls
# ----------------------------------------------------------------------------
@dataclass
class Trainer:
    """create / forward / backward / step / zero_grad on the oracle side."""
    cfg: Config
    seed: int
    params: dict = field(default=None)
    grads: dict = field(default=None)
    m: dict = field(default=None)
    v: dict = field(default=None)
    t: int = 0
    cache: dict = field(default=None)

    def __post_init__(self):
        if self.params is None:
            self.params = init_params(self.cfg, self.seed)
        self.grads = zero_grads(self.params)
        self.m = zero_grads(self.params)
        self.v = zero_grads(self.params)

    def forward(self, tokens, targets=None):
        loss, logits, self.cache = forward(self.params, self.cfg, tokens, targets)
        return loss, logits

    def backward(self):
        backward(self.params, self.cfg, self.cache, self.grads)

    def step(self, lr, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, clip=1.0):
        norm = clip_grads(self.grads, clip)
        self.t += 1
        shapes = dict(param_shapes(self.cfg))
        for name in self.params:
            adamw_update(self.params[name], self.grads[name], self.m[name], self.v[name],
                         self.t, lr, beta1, beta2, eps, weight_decay, decays(name, shapes[name]))
        return norm

    def zero_grad(self):
        for g in self.grads.values():
            g[...] = 0.0
