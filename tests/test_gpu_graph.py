"""One optimizer step (forward, backward, clip + AdamW, zero_grad) captured into
a CUDA graph and replayed gives the same loss, parameters and Adam moments, bit
for bit, as the same steps run eagerly. Every launch of the step goes to the
model's stream or to the library's second stream, which is forked from and
joined back to it by events, and none of these calls synchronises the host
when no host loss or norm is asked for; so one stream capture records the
whole step, the weight-gradient branch and the grouped AdamW included, and a
replay is one launch from the host."""
import numpy as np
import pytest
import torch

import synthdata
from decoder_only_transformer_06_b300 import gpt2
from gpu_helpers import dev, gpu_cfg, oracle_cfg
from oracle import CONFIGS

pytestmark = pytest.mark.gpu


def _step(m, x, y, lr):
    m.forward(x, y, sync_loss=False)
    m.backward()
    m.step(lr, sync_norm=False)
    m.zero_grad()
    m.join()                # the second stream's AdamW and zero_grad rejoin the model's stream


@pytest.mark.parametrize("precision", [gpt2.GPT2_FP32, gpt2.GPT2_BF16])
def test_captured_step_replays_bit_exactly(precision):
    c = oracle_cfg(CONFIGS["char"], batch_size=4, n_layer=2)
    x, y = synthdata.markov_batch(65, c.batch_size, c.seq_len, 1)
    xd, yd = dev(x), dev(y)
    lr = 1e-3
    s = torch.cuda.Stream()
    eager = gpt2.GPT2(gpu_cfg(c, precision), seed=3, stream=s)
    graphed = gpt2.GPT2(gpu_cfg(c, precision), seed=3, stream=s)
    try:
        # one eager step on both first: the kernels' one-time set-up (attributes,
        # occupancy queries, the event pool) happens outside the capture
        for m in (eager, graphed):
            _step(m, xd, yd, lr)
            m.sync()
        for _ in range(2):
            _step(eager, xd, yd, lr)
        eager.sync()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s, capture_error_mode="relaxed"):
            _step(graphed, xd, yd, lr)
        for _ in range(2):
            with torch.cuda.stream(s):
                g.replay()
        s.synchronize()
        graphed.sync()
        assert graphed.loss() == eager.loss()
        for which in (gpt2.GPT2_PARAM, gpt2.GPT2_ADAM_M, gpt2.GPT2_ADAM_V):
            a, b = eager.state(which), graphed.state(which)
            for n in a:
                assert np.array_equal(a[n], b[n]), (which, n)
        # and the graph really ran: two replays moved the parameters past the
        # one eager step both models share
        one_step = gpt2.GPT2(gpu_cfg(c, precision), seed=3, stream=s)
        _step(one_step, xd, yd, lr)
        one_step.sync()
        p1, pg = one_step.state(gpt2.GPT2_PARAM), graphed.state(gpt2.GPT2_PARAM)
        assert any(not np.array_equal(p1[n], pg[n]) for n in p1)
        one_step.close()
    finally:
        eager.close()
        graphed.close()
