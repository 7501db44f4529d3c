"""ctypes binding of libgpt2_b300.so (the C ABI declared in include/gpt2.h).

Argument marshalling only: every step of the training iteration runs in the
library's CUDA kernels. Device buffers are passed as torch tensors (their
data_ptr()), streams as torch.cuda streams. There is no CPU fallback: if the
shared library is missing, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgpt2_b300.so")

GPT2_OK = 0
GPT2_EINVAL = -1
GPT2_ENOMEM = -2
GPT2_ECUDA = -3
GPT2_ESTATE = -4
GPT2_ERANGE = -5
GPT2_ETIMEOUT = -6
GPT2_ENONFINITE = -7
GPT2_FP32 = 0
GPT2_BF16 = 1
GPT2_PARAM, GPT2_GRAD, GPT2_ADAM_M, GPT2_ADAM_V = 0, 1, 2, 3

_ERRNAMES = {
    GPT2_EINVAL: "EINVAL", GPT2_ENOMEM: "ENOMEM", GPT2_ECUDA: "ECUDA", GPT2_ESTATE: "ESTATE",
    GPT2_ERANGE: "ERANGE", GPT2_ETIMEOUT: "ETIMEOUT", GPT2_ENONFINITE: "ENONFINITE",
}


class GPT2Error(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{_ERRNAMES.get(code, code)}: {msg}")
        self.code = code


class gpt2_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "n_layer", "n_head", "d_model", "vocab_size", "padded_vocab", "block_size",
        "batch_size", "seq_len", "grad_accum_steps", "precision")]


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it with `python -m decoder_only_transformer_06_b300.build`")
    lib = ctypes.CDLL(path)
    P, I, I64, F, D, U64 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                           ctypes.c_double, ctypes.c_uint64)
    FP = ctypes.POINTER(ctypes.c_float)
    sig = {
        "gpt2_create": (I, [ctypes.POINTER(gpt2_config), U64, ctypes.POINTER(P)]),
        "gpt2_destroy": (None, [P]),
        "gpt2_set_stream": (I, [P, P]),
        "gpt2_forward": (I, [P, P, P, FP]),
        "gpt2_backward": (I, [P]),
        "gpt2_forward_last": (I, [P, P, I, P]),
        "gpt2_decode_step": (I, [P, P, I, P]),
        "gpt2_step": (I, [P, F, F, F, F, F, F, FP]),
        "gpt2_zero_grad": (I, [P]),
        "gpt2_lr_schedule": (D, [I64, I64, I64, D, D]),
        "gpt2_sync": (I, [P]),
        "gpt2_get_loss": (I, [P, FP]),
        "gpt2_get_loss_async": (I, [P, P]),
        "gpt2_set_wait_limit": (I, [P, ctypes.c_uint]),
        "gpt2_join": (I, [P]),
        "gpt2_num_tensors": (I, [P]),
        "gpt2_tensor_info": (I, [P, I, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(I),
                                 ctypes.POINTER(I64), ctypes.POINTER(I)]),
        "gpt2_copy_tensor": (I, [P, I, I, FP]),
        "gpt2_set_tensor": (I, [P, I, I, FP]),
        "gpt2_copy_logits": (I, [P, I64, I64, FP]),
        "gpt2_copy_row_losses": (I, [P, I64, I64, FP]),
        "gpt2_num_params": (I64, [P, I, I]),
        "gpt2_save": (I, [P, ctypes.c_char_p]),
        "gpt2_load": (I, [P, ctypes.c_char_p]),
        "gpt2_host_init_tensor": (I, [ctypes.POINTER(gpt2_config), U64, I, FP]),
        "gpt2_profile": (I, [P, I]),
        "gpt2_profile_count": (I, [P]),
        "gpt2_profile_entry": (I, [P, I, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(I64),
                                   ctypes.POINTER(I64), ctypes.POINTER(D), ctypes.POINTER(D),
                                   ctypes.POINTER(D)]),
        "gpt2_last_error": (ctypes.c_char_p, [P]),
        "gpt2_version": (ctypes.c_char_p, []),
        "gpt2_op_gemm_bf16": (I, [I, I, I, P, I64, I, P, I64, I, P, P, P, I64, I, P]),
        "gpt2_op_gemm_bf16_gelu": (I, [I, I, I, P, I64, I, P, I64, I, P, I, P, P, I64, P]),
        "gpt2_op_sync": (I, [P]),
        "gpt2_op_set_wait_limit": (I, [ctypes.c_uint]),
        "gpt2_op_sample": (I, [P, I, I, I64, F, I, P, P, P, I, I, P]),
        "gpt2_op_attention_fwd": (I, [I, I, I, I, I, P, P, P, P]),
        "gpt2_op_attention_bwd": (I, [I, I, I, I, I, P, P, P, P, P, P, P]),
        "gpt2_op_attention_bwd_noalloc": (I, [I, I, I, I, I, P, P, P, P, P, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = load_library()


def lib() -> ctypes.CDLL:
    return _lib


def _check(code: int, model=None):
    if code != GPT2_OK:
        raise GPT2Error(code, _lib.gpt2_last_error(model).decode())


def _fp(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


def _stream_ptr(stream) -> int | None:
    if stream is None:
        return None
    return int(getattr(stream, "cuda_stream", stream))


@dataclass
class Config:
    n_layer: int
    n_head: int
    d_model: int
    vocab_size: int
    block_size: int
    batch_size: int
    seq_len: int
    padded_vocab: int = 0
    grad_accum_steps: int = 1
    precision: int = GPT2_BF16

    def to_c(self) -> gpt2_config:
        return gpt2_config(self.n_layer, self.n_head, self.d_model, self.vocab_size,
                           self.padded_vocab, self.block_size, self.batch_size, self.seq_len,
                           self.grad_accum_steps, self.precision)

    @property
    def Vp(self) -> int:
        return self.padded_vocab or ((self.vocab_size + 127) // 128) * 128


def version() -> str:
    return _lib.gpt2_version().decode()


def lr_schedule(it, warmup, horizon, lr_max, lr_min) -> float:
    return _lib.gpt2_lr_schedule(it, warmup, horizon, lr_max, lr_min)


def host_init_tensor(cfg: Config, seed: int, k: int, numel: int) -> np.ndarray:
    out = np.empty(numel, dtype=np.float32)
    c = cfg.to_c()
    _check(_lib.gpt2_host_init_tensor(ctypes.byref(c), seed, k, _fp(out)))
    return out


class GPT2:
    """A model on the current CUDA device (gpt2_create ... gpt2_destroy)."""

    def __init__(self, cfg: Config, seed: int = 1337, stream=None):
        self.cfg = cfg
        self._c = cfg.to_c()
        h = ctypes.c_void_p()
        _check(_lib.gpt2_create(ctypes.byref(self._c), seed, ctypes.byref(h)))
        self.h = h
        self.stream = None           # the legacy default stream until set_stream
        if stream is not None:
            self.set_stream(stream)
        self._info = [self.tensor_info(i) for i in range(self.num_tensors())]
        self.names = [i[0] for i in self._info]

    def close(self):
        if getattr(self, "h", None):
            _lib.gpt2_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _ck(self, code):
        _check(code, self.h)

    def set_stream(self, stream):
        self._ck(_lib.gpt2_set_stream(self.h, _stream_ptr(stream)))
        self.stream = stream

    def forward(self, tokens, targets=None, sync_loss: bool = True):
        """tokens, targets: int32 CUDA tensors [B*T] (or [B, T]). Returns the
        loss (float) when targets are given and sync_loss, else None."""
        loss = ctypes.c_float(float("nan"))
        want = targets is not None and sync_loss
        self._ck(_lib.gpt2_forward(self.h, ctypes.c_void_p(tokens.data_ptr()),
                                   ctypes.c_void_p(targets.data_ptr()) if targets is not None else None,
                                   ctypes.byref(loss) if want else None))
        return loss.value if want else None

    def forward_last(self, tokens, t: int, logits_out):
        """Generation's forward: logits of position t-1 of each of the B
        sequences into logits_out (fp32 CUDA tensor [B, V]); tokens: int32 CUDA
        tensor [B*T] (positions >= t are ignored by causality)."""
        self._ck(_lib.gpt2_forward_last(self.h, ctypes.c_void_p(tokens.data_ptr()), int(t),
                                        ctypes.c_void_p(logits_out.data_ptr())))

    def decode_step(self, tokens, t: int, logits_out):
        """One step with the key/value cache: logits of position t-1 of each
        sequence into logits_out (fp32 CUDA tensor [B, V]); tokens: int32 CUDA
        tensor [B], the token at position t-1 of every sequence (positions
        0..t-2 cached by forward_last or earlier decode steps)."""
        self._ck(_lib.gpt2_decode_step(self.h, ctypes.c_void_p(tokens.data_ptr()), int(t),
                                       ctypes.c_void_p(logits_out.data_ptr())))

    def backward(self):
        self._ck(_lib.gpt2_backward(self.h))

    def step(self, lr, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, clip=1.0,
             sync_norm: bool = True):
        n = ctypes.c_float(float("nan"))
        self._ck(_lib.gpt2_step(self.h, lr, beta1, beta2, eps, weight_decay, clip,
                                ctypes.byref(n) if sync_norm else None))
        return n.value if sync_norm else None

    def zero_grad(self):
        self._ck(_lib.gpt2_zero_grad(self.h))

    def sync(self):
        self._ck(_lib.gpt2_sync(self.h))

    def join(self):
        """The model's stream waits for the library's second stream (no host sync)."""
        self._ck(_lib.gpt2_join(self.h))

    def set_wait_limit(self, cycles: int):
        """Testing hook: bounded-wait limit (SM cycles; 0 = default) of the
        model's single-CTA tensor-core kernels."""
        self._ck(_lib.gpt2_set_wait_limit(self.h, int(cycles)))

    def loss(self) -> float:
        v = ctypes.c_float()
        self._ck(_lib.gpt2_get_loss(self.h, ctypes.byref(v)))
        return v.value

    def loss_async(self, out) -> None:
        """Enqueue a copy of the last forward's loss into out (a float32 CPU
        tensor of one element, pinned for the copy to be asynchronous) on the
        model's stream; it is valid after the next sync."""
        self._ck(_lib.gpt2_get_loss_async(self.h, ctypes.c_void_p(out.data_ptr())))

    def num_tensors(self) -> int:
        return _lib.gpt2_num_tensors(self.h)

    def tensor_info(self, i):
        name = ctypes.c_char_p()
        nd = ctypes.c_int()
        shape = (ctypes.c_int64 * 2)()
        dec = ctypes.c_int()
        self._ck(_lib.gpt2_tensor_info(self.h, i, ctypes.byref(name), ctypes.byref(nd), shape,
                                       ctypes.byref(dec)))
        shp = (shape[0], shape[1]) if nd.value == 2 else (shape[0],)
        return name.value.decode(), shp, bool(dec.value)

    def get(self, i_or_name, which=GPT2_PARAM) -> np.ndarray:
        i = self.names.index(i_or_name) if isinstance(i_or_name, str) else i_or_name
        shape = self._info[i][1]
        out = np.empty(int(np.prod(shape)), dtype=np.float32)
        self._ck(_lib.gpt2_copy_tensor(self.h, i, which, _fp(out)))
        return out.reshape(shape)

    def set(self, i_or_name, value, which=GPT2_PARAM):
        i = self.names.index(i_or_name) if isinstance(i_or_name, str) else i_or_name
        a = np.ascontiguousarray(np.asarray(value, dtype=np.float32).reshape(-1))
        if a.size != int(np.prod(self._info[i][1])):
            raise ValueError("size mismatch")
        self._ck(_lib.gpt2_set_tensor(self.h, i, which, _fp(a)))

    def state(self, which=GPT2_PARAM) -> dict:
        return {n: self.get(i, which) for i, n in enumerate(self.names)}

    def save(self, path):
        """Checkpoint: parameters, Adam moments and step counter (gpt2_save)."""
        self._ck(_lib.gpt2_save(self.h, str(path).encode()))

    def load(self, path):
        """Resume from a checkpoint written by save() for the same config."""
        self._ck(_lib.gpt2_load(self.h, str(path).encode()))

    def logits(self, row0=0, nrows=None) -> np.ndarray:
        M = self.cfg.batch_size * self.cfg.seq_len
        nrows = M - row0 if nrows is None else nrows
        out = np.empty((nrows, self.cfg.vocab_size), dtype=np.float32)
        self._ck(_lib.gpt2_copy_logits(self.h, row0, nrows, _fp(out)))
        return out

    def row_losses(self, row0=0, nrows=None) -> np.ndarray:
        M = self.cfg.batch_size * self.cfg.seq_len
        nrows = M - row0 if nrows is None else nrows
        out = np.empty(nrows, dtype=np.float32)
        self._ck(_lib.gpt2_copy_row_losses(self.h, row0, nrows, _fp(out)))
        return out

    def profile(self, on: bool = True):
        """Clear the per-site counters and switch CUDA-event timing on/off."""
        self._ck(_lib.gpt2_profile(self.h, int(on)))

    def profile_report(self) -> list:
        """Per-site totals since the last profile() call: dicts with name,
        calls, kernels, ms, flops, bytes (synchronises)."""
        n = _lib.gpt2_profile_count(self.h)
        if n < 0:
            self._ck(n)
        out = []
        for i in range(n):
            name = ctypes.c_char_p()
            calls, kern = ctypes.c_int64(), ctypes.c_int64()
            ms, fl, by = ctypes.c_double(), ctypes.c_double(), ctypes.c_double()
            self._ck(_lib.gpt2_profile_entry(self.h, i, ctypes.byref(name), ctypes.byref(calls),
                                             ctypes.byref(kern), ctypes.byref(ms), ctypes.byref(fl),
                                             ctypes.byref(by)))
            out.append(dict(name=name.value.decode(), calls=calls.value, kernels=kern.value,
                            ms=ms.value, flops=fl.value, bytes=by.value))
        return out

    def num_params(self, include_wpe=True, padded=False) -> int:
        return _lib.gpt2_num_params(self.h, int(include_wpe), int(padded))


# ------------------------------------------------------------- op-level calls
def op_gemm_bf16(M, N, K, A, lda, a_kmajor, B, ldb, b_kmajor, bias=None, out_bf16=None,
                 out_f32=None, ldd=None, accumulate=False, stream=None):
    ldd = N if ldd is None else ldd
    ptr = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None
    _check(_lib.gpt2_op_gemm_bf16(M, N, K, ptr(A), lda, int(a_kmajor), ptr(B), ldb, int(b_kmajor),
                                  ptr(bias), ptr(out_bf16), ptr(out_f32), ldd, int(accumulate),
                                  _stream_ptr(stream)))


def op_gemm_bf16_gelu(M, N, K, A, lda, a_kmajor, B, ldb, b_kmajor, out, out2_or_aux, bias=None,
                      backward=False, ldd=None, stream=None):
    """GELU epilogues: backward=False writes out = gelu'(A B^T + bias) and
    out2_or_aux = gelu(A B^T + bias); backward=True writes out = (A B^T) * aux."""
    ldd = N if ldd is None else ldd
    ptr = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None
    _check(_lib.gpt2_op_gemm_bf16_gelu(M, N, K, ptr(A), lda, int(a_kmajor), ptr(B), ldb,
                                       int(b_kmajor), ptr(bias), int(backward), ptr(out),
                                       ptr(out2_or_aux), ldd, _stream_ptr(stream)))


def op_sync(stream=None):
    """Synchronise the stream; raise GPT2Error(ETIMEOUT) if a bounded device
    wait expired in an op-level call since the last op_sync."""
    _check(_lib.gpt2_op_sync(_stream_ptr(stream)))


def op_sample(logits, temperature, top_k, u, out, ctx=None, t=0, stream=None):
    """One sampling step on the device (gpt2_op_sample): logits fp32 CUDA
    [rows, V] (row-contiguous, stride V), u fp32 CUDA [rows] in [0, 1), out int32
    CUDA [rows]; ctx (int32 CUDA [rows, T] with t tokens per row) receives the
    token at position t, or shifted in at T-1 when t == T."""
    rows, V = logits.shape
    T = ctx.shape[1] if ctx is not None else 0
    ptr = lambda x: ctypes.c_void_p(x.data_ptr()) if x is not None else None
    _check(_lib.gpt2_op_sample(ptr(logits), rows, V, logits.stride(0), float(temperature),
                               int(top_k or 0), ptr(u), ptr(out), ptr(ctx), T, int(t),
                               _stream_ptr(stream)))


def op_set_wait_limit(cycles: int):
    """Testing hook: bounded-wait limit (SM cycles; 0 = default) of the
    op-level calls' single-CTA kernels on the current device."""
    _check(_lib.gpt2_op_set_wait_limit(int(cycles)))


def op_attention_fwd(precision, B, T, H, hs, qkv, out, lse, stream=None):
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())
    _check(_lib.gpt2_op_attention_fwd(precision, B, T, H, hs, ptr(qkv), ptr(out), ptr(lse),
                                      _stream_ptr(stream)))


def op_attention_bwd(precision, B, T, H, hs, qkv, out, lse, dout, dqkv, scratch, stream=None):
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())
    _check(_lib.gpt2_op_attention_bwd(precision, B, T, H, hs, ptr(qkv), ptr(out), ptr(lse),
                                      ptr(dout), ptr(dqkv), ptr(scratch), _stream_ptr(stream)))


def op_attention_bwd_noalloc(precision, B, T, H, hs, qkv, out, lse, dout, dqkv, stream=None):
    """gpt2_op_attention_bwd without a scratch argument: the library keeps the
    rowsum scratch in a fixed device array of its own (B*H*T <= 2**20), for
    callers that must not allocate device memory."""
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())
    _check(_lib.gpt2_op_attention_bwd_noalloc(precision, B, T, H, hs, ptr(qkv), ptr(out),
                                              ptr(lse), ptr(dout), ptr(dqkv),
                                              _stream_ptr(stream)))
