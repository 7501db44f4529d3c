"""The C-ABI library without a GPU: it loads, exports every symbol that
include/gpt2.h declares, and its host-only logic (config validation, init,
schedule) agrees with the oracle. No compute call touches a GPU here."""
import ctypes
import math
import os
import re
import subprocess

import numpy as np
import pytest

import synthdata  # noqa: F401  (keeps the import graph of the suite uniform)
from decoder_only_transformer_06_b300 import gpt2
from oracle import CONFIGS
from oracle import gpt2_oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gpt2.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s*(gpt2_[a-z0-9_]+)\s*\(",
                       src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary_calls():
    names = declared_functions()
    for must in ("gpt2_create", "gpt2_forward", "gpt2_backward", "gpt2_step", "gpt2_zero_grad",
                 "gpt2_destroy"):
        assert must in names


def test_library_exports_every_declared_symbol():
    lib = gpt2.lib()
    for n in declared_functions():
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", gpt2.LIB_PATH], capture_output=True,
                         text=True).stdout
    exported = set(re.findall(r"\bT (gpt2_[a-z0-9_]+)", out))
    assert set(declared_functions()) <= exported


def test_version_string():
    assert "sm_103a" in gpt2.version()


def _cfg(name, precision=gpt2.GPT2_BF16, **kw):
    c = CONFIGS[name]
    d = dict(n_layer=c.n_layer, n_head=c.n_head, d_model=c.d_model, vocab_size=c.vocab_size,
             block_size=c.block_size, batch_size=c.batch_size, seq_len=c.seq_len,
             padded_vocab=c.padded_vocab, grad_accum_steps=c.grad_accum_steps, precision=precision)
    d.update(kw)
    return gpt2.Config(**d)


def test_host_init_matches_oracle_tiny_bit_exact():
    cfg = _cfg("tiny", gpt2.GPT2_FP32)
    ref = O.init_params(CONFIGS["tiny"], 1337)
    for k, (name, shape) in enumerate(O.param_shapes(CONFIGS["tiny"])):
        got = gpt2.host_init_tensor(cfg, 1337, k, int(np.prod(shape))).reshape(shape)
        assert np.array_equal(got.astype(np.float64), ref[name]), name


def test_host_init_matches_oracle_gpt2_slices():
    """GPT-2 124M: compare a few whole tensors (wpe, layer-11 projections)."""
    c = CONFIGS["gpt2_124m"]
    cfg = _cfg("gpt2_124m")
    shapes = O.param_shapes(c)
    names = [n for n, _ in shapes]
    for name in ("wpe", "h11.attn_proj.W", "h0.fc.W"):
        k = names.index(name)
        shape = shapes[k][1]
        n = int(np.prod(shape))
        got = gpt2.host_init_tensor(cfg, 7, k, n).astype(np.float64)
        std = 0.02 / math.sqrt(24) if "proj.W" in name else 0.02
        ref = (std * O.init_normals(7, k, n)).astype(np.float32).astype(np.float64)
        mism = np.count_nonzero(got != ref)
        # libm and numpy may differ by an ulp in double; after rounding to fp32
        # that changes a value only rarely, and then by one fp32 ulp
        assert mism <= 2, (name, mism)
        assert np.allclose(got, ref, rtol=2 ** -23, atol=0)


def test_lr_schedule_matches_oracle():
    for it in (0, 1, 500, 714, 715, 716, 5000, 19073, 19074, 30000):
        assert abs(gpt2.lr_schedule(it, 715, 19073, 6e-4, 6e-5) -
                   O.lr_schedule(it, 715, 19073, 6e-4, 6e-5)) < 1e-15
    assert abs(gpt2.lr_schedule(301000, 2000, 600000, 6e-4, 6e-5) - 3.3e-4) < 1e-12


@pytest.mark.parametrize("bad", [
    dict(d_model=65),                       # not a multiple of n_head / 32
    dict(seq_len=2048),                     # beyond block_size
    dict(padded_vocab=50000),               # below vocab_size
    dict(padded_vocab=50260),               # not a multiple of 64
    dict(batch_size=0),
    dict(precision=7),
    dict(n_head=8),                         # bf16 path needs head size 64 (768/8 = 96)
])
def test_create_rejects_bad_configs_without_touching_the_gpu(bad):
    cfg = _cfg("gpt2_124m", **bad)
    c = cfg.to_c()
    h = ctypes.c_void_p()
    r = gpt2.lib().gpt2_create(ctypes.byref(c), 1, ctypes.byref(h))
    assert r == gpt2.GPT2_EINVAL and not h.value
    assert gpt2.lib().gpt2_last_error(None)


def test_injected_allocation_failure_is_reported(monkeypatch):
    """Host-side fault injection: the first device allocation of gpt2_create
    fails (before any CUDA call); the call returns ENOMEM with no model and a
    message naming the injected failure."""
    monkeypatch.setenv("GPT2_FAIL_ALLOC_AT", "0")
    c = _cfg("tiny", precision=gpt2.GPT2_FP32).to_c()     # head size 16: the fp32-math path
    h = ctypes.c_void_p()
    r = gpt2.lib().gpt2_create(ctypes.byref(c), 1, ctypes.byref(h))
    assert r == gpt2.GPT2_ENOMEM and not h.value
    assert b"injected allocation failure at allocation 0" in gpt2.lib().gpt2_last_error(None)


def test_null_arguments_are_rejected():
    L = gpt2.lib()
    assert L.gpt2_create(None, 1, None) == gpt2.GPT2_EINVAL
    assert L.gpt2_forward(None, None, None, None) == gpt2.GPT2_EINVAL
    assert L.gpt2_backward(None) == gpt2.GPT2_EINVAL
    assert L.gpt2_step(None, 1e-3, 0.9, 0.95, 1e-8, 0.1, 1.0, None) == gpt2.GPT2_EINVAL
    assert L.gpt2_zero_grad(None) == gpt2.GPT2_EINVAL
    assert L.gpt2_save(None, b"/dev/null") == gpt2.GPT2_EINVAL
    assert L.gpt2_load(None, b"/dev/null") == gpt2.GPT2_EINVAL
    L.gpt2_destroy(None)
