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


def adamw_param_diff(p_gpu, p_orc, g_gpu, g_orc):
    """Max |p_gpu - p_orc| over elements whose gradients agree in sign, and the
    number of elements whose signs differ (a first AdamW step moves every
    element by about lr whatever |g|, so a sign flip at the noise floor moves
    it by 2 lr)."""
    p_gpu, p_orc = np.asarray(p_gpu, np.float64), np.asarray(p_orc, np.float64)
    agree = np.sign(g_gpu) == np.sign(g_orc)
    d = np.abs(p_gpu - p_orc)
    return float(d[agree].max()) if agree.any() else 0.0, int((~agree).sum())
