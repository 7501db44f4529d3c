"""CPU oracle for the GPT-2 training step.

TEST INFRASTRUCTURE ONLY: the plain fp64 reference that the CUDA library is
checked against. Only the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import it. It shares no code with the library
and imports nothing from it; the only module both sides use is ``synthdata``
(seeded token streams, no model arithmetic).

Parity pins (what checks the oracle itself, independently of the CUDA path):
see tests/test_oracle_pins.py. Every function here is pinned; none is marked
"parity unpinned".
"""
from .gpt2_oracle import (  # noqa: F401
    Config, Trainer, adamw_update, attention_bwd, attention_fwd, backward,
    causal_lse, causal_softmax, clip_grads, decays, forward, gelu_tanh, gelu_tanh_grad,
    global_grad_norm, init_normals, init_params, layernorm_bwd, layernorm_fwd,
    lr_schedule, num_params, param_shapes, sample_tokens, zero_grads,
)

# The five workloads the method is exercised on (tiny fp32 check, character
# model, GPT-2 124M, 124M with 32-way accumulation, 24-layer/1024-wide).
CONFIGS = {
    "tiny": Config(n_layer=2, n_head=4, d_model=64, vocab_size=65, block_size=64,
                   batch_size=4, seq_len=64),
    "char": Config(n_layer=6, n_head=6, d_model=384, vocab_size=65, block_size=256,
                   batch_size=64, seq_len=256),
    "gpt2_124m": Config(n_layer=12, n_head=12, d_model=768, vocab_size=50257,
                        padded_vocab=50304, block_size=1024, batch_size=16, seq_len=1024),
    "gpt2_124m_accum32": Config(n_layer=12, n_head=12, d_model=768, vocab_size=50257,
                                padded_vocab=50304, block_size=1024, batch_size=16,
                                seq_len=1024, grad_accum_steps=32),
    "gpt2_24l_1024d": Config(n_layer=24, n_head=16, d_model=1024, vocab_size=50257,
                             padded_vocab=50304, block_size=1024, batch_size=8, seq_len=1024),
}
