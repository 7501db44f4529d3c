"""Shared helpers for the GPU parity tests (no oracle arithmetic here: only
config conversion, device transfer and comparison metrics)."""
import numpy as np
import torch

from decoder_only_transformer_06_b300 import gpt2
from oracle import gpt2_oracle as O


def gpu_cfg(c: O.Config, precision, **kw) -> gpt2.Config:
    d = dict(n_layer=c.n_layer, n_head=c.n_head, d_model=c.d_model, vocab_size=c.vocab_size,
             block_size=c.block_size, batch_size=c.batch_size, seq_len=c.seq_len,
             padded_vocab=c.padded_vocab, grad_accum_steps=c.grad_accum_steps, precision=precision)
    d.update(kw)
    return gpt2.Config(**d)


def oracle_cfg(c: O.Config, **kw) -> O.Config:
    return O.Config(**{**c.__dict__, **kw})


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a.reshape(-1)).astype(np.int32)).cuda()


def rel_l2(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / nb) if nb > 0 else float(np.linalg.norm(a))


def cosine(a, b) -> float:
    a = np.asarray(a, dtype=np.float64).reshape(-1)
    b = np.asarray(b, dtype=np.float64).reshape(-1)
    na, nb = np.linalg.norm(a), np.linalg.norm(b)
    if na == 0 and nb == 0:
        return 1.0
    return float(a @ b / (na * nb))


def adamw_param_check(p_gpu, p_orc, g_gpu, g_orc, fp32: bool, coef: float = 1.0):
    """Post-AdamW parameter comparison (first step, lr ~1e-3).

    A first AdamW step moves an element by lr * g / (|g| + eps) (plus the
    identical decay), i.e. by about lr whatever |g|, so:
      * where the GPU and oracle gradients agree in sign, |p_gpu - p_orc| is
        returned as `agree_max` (bf16 bound 1e-3; for fp32 only elements whose
        clipped gradient coef*|g| (the gradient AdamW sees; coef = the clip
        coefficient) is >= 100*eps are taken, because the step's sensitivity
        lr*eps/(|g|+eps)^2 grows without bound as |g| nears eps and an fp32
        gradient there carries relative error);
      * a sign flip moves an element by up to 2 lr; `big_flips` counts flips
        among elements whose oracle gradient is large (> 0.1 * the tensor's RMS
        and > eps), where none should occur.
    Returns (agree_max, big_flips, all_max)."""
    p_gpu, p_orc = np.asarray(p_gpu, np.float64), np.asarray(p_orc, np.float64)
    g_gpu, g_orc = np.asarray(g_gpu, np.float64), np.asarray(g_orc, np.float64)
    d = np.abs(p_gpu - p_orc)
    agree = np.sign(g_gpu) == np.sign(g_orc)
    sel = agree & (coef * np.abs(g_orc) >= 1e-6) if fp32 else agree
    agree_max = float(d[sel].max()) if sel.any() else 0.0
    rms = float(np.sqrt(np.mean(g_orc ** 2))) if g_orc.size else 0.0
    big = (np.abs(g_orc) > 0.1 * rms) & (np.abs(g_orc) > 1e-8)
    big_flips = int(np.count_nonzero(big & ~agree))
    return agree_max, big_flips, float(d.max())


def oracle_adamw_on(params0, grads, lr, t=1, beta1=0.9, beta2=0.95, eps=1e-8, wd=0.1, clip=1.0):
    """The oracle's clip + AdamW applied to given gradients (the optimizer in
    isolation: fed the GPU's own gradients it must reproduce the GPU's update)."""
    from oracle import gpt2_oracle as O
    g = {n: np.asarray(a, np.float64).copy() for n, a in grads.items()}
    O.clip_grads(g, clip)
    out = {}
    for n, p0 in params0.items():
        p = np.asarray(p0, np.float64).copy()
        m = np.zeros_like(p)
        v = np.zeros_like(p)
        O.adamw_update(p, g[n], m, v, t, lr, beta1, beta2, eps, wd, p.ndim >= 2)
        out[n] = p
    return out
