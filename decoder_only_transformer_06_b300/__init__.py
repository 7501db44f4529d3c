"""B300-native GPT-2 training step: CUDA kernels for sm_103a behind a C ABI
(include/gpt2.h), with a thin ctypes binding.

    from decoder_only_transformer_06_b300 import gpt2
    m = gpt2.GPT2(gpt2.Config(n_layer=12, n_head=12, d_model=768, vocab_size=50257,
                              padded_vocab=50304, block_size=1024, batch_size=16,
                              seq_len=1024, precision=gpt2.GPT2_BF16))
    loss = m.forward(tokens, targets); m.backward(); m.step(lr=6e-4); m.zero_grad()

Importing ``gpt2`` loads libgpt2_b300.so and fails loudly if it is missing.
"""

__all__ = ["gpt2", "build"]
