"""Op-level parity: each tensor-core / attention kernel against the oracle's
definition (fp64 on the same bf16-rounded inputs), through the C ABI."""
import math

import numpy as np
import pytest
import torch

from decoder_only_transformer_06_b300 import gpt2
from oracle import gpt2_oracle as O

from gpu_helpers import rel_l2

pytestmark = pytest.mark.gpu


def _gemm_case(M, N, K, ak, bk, seed):
    g = torch.Generator().manual_seed(seed)
    A = torch.randn(M, K, generator=g, dtype=torch.float32).bfloat16()
    B = torch.randn(N, K, generator=g, dtype=torch.float32).bfloat16()
    a_mem = A if ak else A.t().contiguous()
    b_mem = B if bk else B.t().contiguous()
    lda = K if ak else M
    ldb = K if bk else N
    ref = A.double().numpy() @ B.double().numpy().T
    return a_mem.cuda(), lda, b_mem.cuda(), ldb, ref


SHAPES = [(128, 128, 64), (256, 512, 128), (384, 768, 768), (200, 96, 80), (136, 264, 200),
          (128, 2304, 64), (1024, 3072, 192), (256, 50304, 64)]


@pytest.mark.parametrize("ak,bk", [(1, 1), (1, 0), (0, 1), (0, 0)])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_gemm_bf16_fp32_out(M, N, K, ak, bk):
    a, lda, b, ldb, ref = _gemm_case(M, N, K, ak, bk, M * 7 + N * 3 + K + 10 * ak + bk)
    out = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    gpt2.op_gemm_bf16(M, N, K, a, lda, ak, b, ldb, bk, out_f32=out)
    gpt2.op_sync()
    got = out.cpu().double().numpy()
    # fp32 accumulation of exact bf16 products: error ~ sqrt(K) * 2^-24 * |terms|
    assert np.abs(got - ref).max() <= 1e-4 * math.sqrt(K) * 4, (M, N, K, ak, bk)


# N = 384 runs 128-wide single-CTA tiles, N = 768 256-wide tiles on CTA pairs
# (M = 320 leaves the second pair tile more than half empty)
@pytest.mark.parametrize("N", [384, 768])
@pytest.mark.parametrize("ak,bk", [(1, 1), (1, 0), (0, 0)])
def test_gemm_bf16_bias_bf16_out_and_accumulate(ak, bk, N):
    M, K = 320, 256
    a, lda, b, ldb, ref = _gemm_case(M, N, K, ak, bk, 5 + N)
    bias = torch.randn(N, dtype=torch.float32).cuda()
    out = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    gpt2.op_gemm_bf16(M, N, K, a, lda, ak, b, ldb, bk, bias=bias, out_bf16=out)
    acc = torch.ones(M, N, dtype=torch.float32, device="cuda")
    gpt2.op_gemm_bf16(M, N, K, a, lda, ak, b, ldb, bk, out_f32=acc, accumulate=True)
    gpt2.op_sync()
    r = ref + bias.cpu().double().numpy()[None, :]
    got = out.cpu().double().numpy()
    assert np.all(np.abs(got - r) <= 2 ** -8 * np.abs(r) + 1e-3 * math.sqrt(K))
    assert np.abs(acc.cpu().double().numpy() - (ref + 1.0)).max() <= 4e-4 * math.sqrt(K)


def _gelu_bound(pre, ref, deriv):
    """Per-element bound for the GELU epilogues: bf16 rounding of the output
    (2^-9 relative, 2^-8 allowed), fp32 accumulation of the products (K * 2^-24
    relative to sum |a b|, below 1e-5 here) and the hardware tanh (absolute
    error e = 2^-10.9 in t): gelu = 0.5 x (1 + t) moves by 0.5 |x| e, and
    gelu' = 0.5 (1 + t) + 0.5 x (1 - t^2) u' by 0.5 e + |x| |t| e u', with
    u' = sqrt(2/pi) (1 + 3 * 0.044715 x^2)."""
    e = 2.0 ** -10.9
    hx = 0.5 * np.abs(pre)
    if deriv:
        up = 0.7978845608028654 * (1.0 + 3.0 * 0.044715 * pre * pre)
        t = np.tanh(0.7978845608028654 * (pre + 0.044715 * pre ** 3))
        ta = 0.5 * e + 2.0 * hx * np.abs(t) * e * up
    else:
        ta = hx * e
    return 2.0 ** -8 * np.abs(ref) + ta + 1e-5


# N = 768 runs on CTA pairs, N = 384 on single CTAs; M = 320 leaves the last
# tile partly empty; K-major and MN-major B (the forward and the dX layouts)
@pytest.mark.parametrize("N", [384, 768])
@pytest.mark.parametrize("bk", [1, 0])
def test_gemm_gelu_epilogues(N, bk):
    M, K = 320, 256
    g = torch.Generator().manual_seed(N + bk)
    A = torch.randn(M, K, generator=g, dtype=torch.float32).bfloat16()
    # weights of std 0.1 keep pre-activations around N(0, 1.6^2): the range
    # where GELU bends
    Bw = (0.1 * torch.randn(N, K, generator=g, dtype=torch.float32)).bfloat16()
    bias = (0.5 * torch.randn(N, generator=g, dtype=torch.float32))
    b_mem = Bw if bk else Bw.t().contiguous()
    ldb = K if bk else N
    pre = A.double().numpy() @ Bw.double().numpy().T
    # forward: out = gelu'(pre + bias), out2 = gelu(pre + bias)
    d = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    h = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    gpt2.op_gemm_bf16_gelu(M, N, K, A.cuda(), K, 1, b_mem.cuda(), ldb, bk, d, h, bias=bias.cuda())
    # backward: out = pre * aux, with an arbitrary bf16 aux
    aux = torch.randn(M, N, generator=g, dtype=torch.float32).bfloat16()
    y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    gpt2.op_gemm_bf16_gelu(M, N, K, A.cuda(), K, 1, b_mem.cuda(), ldb, bk, y, aux.cuda(), backward=True)
    gpt2.op_sync()
    x = pre + bias.double().numpy()[None, :]
    ref_h, ref_d = O.gelu_tanh(x), O.gelu_tanh_grad(x)
    got_h, got_d = h.cpu().double().numpy(), d.cpu().double().numpy()
    assert np.all(np.abs(got_h - ref_h) <= _gelu_bound(x, ref_h, False)), (N, bk)
    assert np.all(np.abs(got_d - ref_d) <= _gelu_bound(x, ref_d, True)), (N, bk)
    ref_y = pre * aux.double().numpy()
    got_y = y.cpu().double().numpy()
    assert np.all(np.abs(got_y - ref_y) <= 2.0 ** -8 * np.abs(ref_y) + 1e-5 * np.abs(aux.double().numpy()) * math.sqrt(K)), (N, bk)


def _attn_inputs(B, T, H, hs, seed, dtype):
    g = torch.Generator().manual_seed(seed)
    qkv = torch.randn(B * T, 3 * H * hs, generator=g, dtype=torch.float32)
    dout = torch.randn(B * T, H * hs, generator=g, dtype=torch.float32)
    if dtype == torch.bfloat16:
        qkv, dout = qkv.bfloat16(), dout.bfloat16()
    return qkv, dout


def _oracle_attn(qkv, dout, B, T, H, hs):
    C = H * hs
    x = qkv.double().numpy().reshape(B, T, 3 * C)
    f = lambda t: t.reshape(B, T, H, hs).transpose(0, 2, 1, 3)
    q, k, v = f(x[..., :C]), f(x[..., C:2 * C]), f(x[..., 2 * C:])
    o = O.attention_fwd(q, k, v)
    lse = O.causal_lse(q, k)
    do = f(dout.double().numpy().reshape(B, T, C))
    dq, dk, dv = O.attention_bwd(do, q, k, v)
    m = lambda t: t.transpose(0, 2, 1, 3).reshape(B * T, C)
    return m(o), lse.reshape(B * H * T), np.concatenate([m(dq), m(dk), m(dv)], axis=1)


@pytest.mark.parametrize("precision", [gpt2.GPT2_BF16, gpt2.GPT2_FP32])
@pytest.mark.parametrize("B,T,H", [(2, 256, 2), (1, 200, 3), (3, 64, 1), (2, 1, 2), (1, 1024, 2)])
def test_attention_fwd_bwd(precision, B, T, H):
    hs = 64
    dt = torch.bfloat16 if precision == gpt2.GPT2_BF16 else torch.float32
    qkv, dout = _attn_inputs(B, T, H, hs, B * 1000 + T + H, dt)
    o_ref, lse_ref, d_ref = _oracle_attn(qkv, dout, B, T, H, hs)
    C = H * hs
    q_d, do_d = qkv.cuda(), dout.cuda()
    out = torch.empty(B * T, C, dtype=dt, device="cuda")
    lse = torch.empty(B * H * T, dtype=torch.float32, device="cuda")
    dqkv = torch.empty(B * T, 3 * C, dtype=dt, device="cuda")
    scratch = torch.empty(B * H * T, dtype=torch.float32, device="cuda")
    gpt2.op_attention_fwd(precision, B, T, H, hs, q_d, out, lse)
    gpt2.op_attention_bwd(precision, B, T, H, hs, q_d, out, lse, do_d, dqkv, scratch)
    gpt2.op_sync()
    o = out.float().cpu().double().numpy()
    l = lse.cpu().double().numpy()
    d = dqkv.float().cpu().double().numpy()
    if precision == gpt2.GPT2_FP32:
        assert np.abs(o - o_ref).max() < 1e-5
        assert np.abs(l - lse_ref).max() < 1e-5
        assert rel_l2(d, d_ref) < 1e-5
    else:
        assert np.abs(o - o_ref).max() < 3e-2
        assert np.abs(l - lse_ref).max() < 2e-3
        for part in range(3):
            sl = slice(part * C, (part + 1) * C)
            assert rel_l2(d[:, sl], d_ref[:, sl]) < 2e-2, part


def test_attention_rejects_unsupported_head_size():
    qkv = torch.zeros(64, 3 * 96, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(64, 96, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(64, dtype=torch.float32, device="cuda")
    with pytest.raises(gpt2.GPT2Error):
        gpt2.op_attention_fwd(gpt2.GPT2_BF16, 1, 64, 1, 96, qkv, out, lse)
