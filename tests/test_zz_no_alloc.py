"""The allocation-free attention backward (gpt2_op_attention_bwd_noalloc).

Some callers may not allocate device memory at all: a plugin whose host
application owns every device allocation, or a service that forbids
cudaMalloc once it has started. For them the library offers this one variant
of the attention backward, whose rowsum scratch is a fixed array compiled into
the library instead of a buffer the caller allocates. These tests call it
through the C ABI and check it against gpt2_op_attention_bwd (which takes a
caller-allocated scratch) on two calls in a row, so that anything the first
call leaves in the shared array cannot leak into the second.

This file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest

from decoder_only_transformer_06_b300 import gpt2


def _inputs(B, T, H, hs, seed, dtype):
    import torch
    g = torch.Generator().manual_seed(seed)
    qkv = torch.randn(B * T, 3 * H * hs, generator=g, dtype=torch.float32).to(dtype)
    dout = torch.randn(B * T, H * hs, generator=g, dtype=torch.float32).to(dtype)
    return qkv.cuda(), dout.cuda()


def _run(precision, B, T, H, hs, seed):
    """dqkv from both entry points on the same inputs."""
    import torch
    dt = torch.bfloat16 if precision == gpt2.GPT2_BF16 else torch.float32
    qkv, dout = _inputs(B, T, H, hs, seed, dt)
    C = H * hs
    out = torch.empty(B * T, C, dtype=dt, device="cuda")
    lse = torch.empty(B * H * T, dtype=torch.float32, device="cuda")
    gpt2.op_attention_fwd(precision, B, T, H, hs, qkv, out, lse)
    ref = torch.full((B * T, 3 * C), float("nan"), dtype=dt, device="cuda")
    scratch = torch.empty(B * H * T, dtype=torch.float32, device="cuda")
    gpt2.op_attention_bwd(precision, B, T, H, hs, qkv, out, lse, dout, ref, scratch)
    got = torch.full((B * T, 3 * C), float("nan"), dtype=dt, device="cuda")
    gpt2.op_attention_bwd_noalloc(precision, B, T, H, hs, qkv, out, lse, dout, got)
    torch.cuda.synchronize()
    return got.float().cpu().numpy(), ref.float().cpu().numpy()


@pytest.mark.gpu
@pytest.mark.parametrize("precision", [gpt2.GPT2_BF16, gpt2.GPT2_FP32])
def test_noalloc_attention_bwd_matches_the_allocating_entry_point(precision):
    # two calls in a row on one device: a larger case, then a smaller ragged
    # one; both entry points run the same kernels on the same inputs, so the
    # outputs must be identical bit for bit
    for B, T, H, seed in ((4, 512, 3, 11), (2, 200, 2, 12)):
        got, ref = _run(precision, B, T, H, 64, seed)
        assert np.all(np.isfinite(got))
        assert np.array_equal(got, ref), (precision, B, T, H)


@pytest.mark.gpu
def test_noalloc_attention_bwd_fills_its_scratch_to_the_limit():
    """B*H*T exactly 2^20 rows: the last row of the fixed array is used."""
    got, ref = _run(gpt2.GPT2_BF16, 1024, 1024, 1, 64, 13)
    assert np.all(np.isfinite(got))
    assert np.array_equal(got, ref)


@pytest.mark.gpu
def test_noalloc_attention_bwd_reports_an_expired_wait():
    """The allocation-free path's kernels record a bounded-wait expiry in the
    library's fixed status word; gpt2_op_sync reports it as ETIMEOUT (and
    allocates nothing to do so). With the default limit back, the next call is
    bit-identical to the allocating entry point."""
    import torch
    B, T, H, hs = 2, 512, 2, 64
    qkv, dout = _inputs(B, T, H, hs, 14, torch.bfloat16)
    C = H * hs
    out = torch.empty(B * T, C, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B * H * T, dtype=torch.float32, device="cuda")
    gpt2.op_attention_fwd(gpt2.GPT2_BF16, B, T, H, hs, qkv, out, lse)
    got = torch.empty(B * T, 3 * C, dtype=torch.bfloat16, device="cuda")
    gpt2.op_sync()
    gpt2.op_set_wait_limit(200)
    try:
        gpt2.op_attention_bwd_noalloc(gpt2.GPT2_BF16, B, T, H, hs, qkv, out, lse, dout, got)
        with pytest.raises(gpt2.GPT2Error) as e:
            gpt2.op_sync()
        assert e.value.code == gpt2.GPT2_ETIMEOUT
    finally:
        gpt2.op_set_wait_limit(0)
    gpt2.op_sync()                      # the report cleared the status
    got2, ref = _run(gpt2.GPT2_BF16, B, T, H, hs, 14)
    assert np.array_equal(got2, ref)


def test_noalloc_attention_bwd_rejects_sizes_beyond_its_scratch():
    """B*H*T above 2^20 is refused before any device work (no GPU needed:
    the pointers are never dereferenced)."""
    fake = ctypes.c_void_p(256)
    rc = gpt2.lib().gpt2_op_attention_bwd_noalloc(gpt2.GPT2_BF16, 16, 1024, 65, 64, fake, fake,
                                                 fake, fake, fake, None)
    assert rc == gpt2.GPT2_EINVAL
    assert b"exceeds the fixed scratch" in gpt2.lib().gpt2_last_error(None)
