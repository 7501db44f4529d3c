"""Failure detection on the GPU in the permitted forms: a bounded device wait
that is made to run out (its limit lowered to a few hundred cycles, so the
wait expires long before the copy or product it waits for lands), and an
allocation failure injected on the host. Nothing here faults, traps or hangs
a GPU: an expired wait makes the kernel record ERR_TIMEOUT, drain its own
in-flight copies and products with the full limit, free its tensor memory and
return, after which the host reads the status and the context stays usable.
"""
import os

import numpy as np
import pytest
import torch

import synthdata
from decoder_only_transformer_06_b300 import gpt2
from oracle import CONFIGS
from oracle import gpt2_oracle as O

from gpu_helpers import cosine, dev, gpu_cfg, oracle_cfg, rel_l2

pytestmark = pytest.mark.gpu

SHORT = 200       # cycles: far below any copy's or product's latency


def _gemm_case(seed=0):
    # N = 128: a single-CTA tile (CTA pairs keep the full limit); K = 16384
    # gives the epilogue warps a main loop of thousands of cycles to wait for
    M, N, K = 256, 128, 16384
    g = torch.Generator(device="cuda").manual_seed(seed)
    A = torch.randn(M, K, device="cuda", generator=g).bfloat16()
    B = torch.randn(N, K, device="cuda", generator=g).bfloat16()
    return M, N, K, A, B


def test_gemm_wait_expires_then_the_next_call_is_correct():
    M, N, K, A, B = _gemm_case()
    out = torch.zeros(M, N, dtype=torch.float32, device="cuda")
    gpt2.op_sync()
    gpt2.op_set_wait_limit(SHORT)
    try:
        gpt2.op_gemm_bf16(M, N, K, A, K, True, B, K, True, out_f32=out)
        with pytest.raises(gpt2.GPT2Error) as e:
            gpt2.op_sync()
        assert e.value.code == gpt2.GPT2_ETIMEOUT
    finally:
        gpt2.op_set_wait_limit(0)
    # the status was cleared by the report; the context works and the next
    # call computes the full product
    gpt2.op_gemm_bf16(M, N, K, A, K, True, B, K, True, out_f32=out)
    gpt2.op_sync()
    ref = A.double() @ B.double().T
    err = (out.double() - ref).abs().max().item()
    assert err <= 1e-3 * ref.abs().max().item(), err


def test_model_wait_expires_then_a_full_step_matches_the_oracle():
    """A bf16 model whose attention and most GEMMs run single-CTA kernels:
    with the short limit its forward reports ETIMEOUT; with the default
    restored, one full step matches the oracle within the bf16 tolerances."""
    c = O.Config(n_layer=2, n_head=2, d_model=128, vocab_size=65, block_size=128,
                 batch_size=2, seq_len=128)
    m = gpt2.GPT2(gpu_cfg(c, gpt2.GPT2_BF16), seed=6)
    x, y = synthdata.uniform_batch(65, c.batch_size, c.seq_len, 61)
    m.set_wait_limit(SHORT)
    with pytest.raises(gpt2.GPT2Error) as e:
        m.forward(dev(x), dev(y))
    assert e.value.code == gpt2.GPT2_ETIMEOUT
    m.set_wait_limit(0)
    m.sync()                                  # nothing left to report
    tr = O.Trainer(c, 6)
    loss = m.forward(dev(x), dev(y))
    lo, _ = tr.forward(x, y)
    assert abs(loss - lo) / lo < 5e-3, (loss, lo)
    m.backward()
    tr.backward()
    g = m.state(gpt2.GPT2_GRAD)
    for n, ref in tr.grads.items():
        if not np.any(ref):
            continue
        assert rel_l2(g[n], ref) <= 2e-2 and cosine(g[n], ref) >= 0.999, n
    m.close()


def test_injected_allocation_failure_frees_everything():
    """GPT2_FAIL_ALLOC_AT=5: the sixth device allocation of gpt2_create fails
    after five succeeded; create returns ENOMEM, the five are freed (device
    free memory back to its level before the call), and the next create
    succeeds and trains."""
    c = oracle_cfg(CONFIGS["gpt2_124m"], n_layer=2, batch_size=1, seq_len=64)
    cfg = gpu_cfg(c, gpt2.GPT2_BF16)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    os.environ["GPT2_FAIL_ALLOC_AT"] = "5"
    try:
        with pytest.raises(gpt2.GPT2Error) as e:
            gpt2.GPT2(cfg, seed=1)
        assert e.value.code == gpt2.GPT2_ENOMEM
        assert "allocation 5" in str(e.value)
    finally:
        del os.environ["GPT2_FAIL_ALLOC_AT"]
    free1 = torch.cuda.mem_get_info()[0]
    # the five arenas held about 0.9 GB; all of it is back
    assert free1 >= free0 - (64 << 20), (free0, free1)
    m = gpt2.GPT2(cfg, seed=1)
    x, y = synthdata.zipf_batch(c.vocab_size, 1, 64, 3)
    loss = m.forward(dev(x), dev(y))
    m.backward()
    assert np.isfinite(loss) and np.isfinite(m.step(lr=6e-4))
    m.close()
