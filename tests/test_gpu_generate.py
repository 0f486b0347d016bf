"""Greedy generation through the C ABI with the decode forward captured in a CUDA
graph ("Tensor parallelism from scratch", tp.py main: 20 greedy tokens after a
prompt), against the oracle's generation loop token by token."""

import numpy as np
import pytest
import torch

import synth
import synth.device as sd
from oracle import forward as of
from oracle import inputs as oi
from tests.gpu_harness import KV_DTYPE, MARGIN, assert_close, model_config

pytestmark = pytest.mark.gpu

LAYERS = 2
STEPS = 20


def _prompts(vocab: int, lens, seed: int):
    rng = np.random.default_rng(seed)
    return [[int(t) for t in rng.integers(0, vocab, size=n)] for n in lens]


def _runner(s: synth.ModelShape, n: int, B: int, capacity: int, max_tokens: int):
    from tensor_transformer_forward_gb300.runner import TPRunner
    r = TPRunner(model_config(s, n), LAYERS, B, capacity, max_tokens)
    for li in range(LAYERS):
        r.load_layer(li, sd.layer_weights(s, li, True))
    r.load_head(sd.head_weights(s, True))
    for kv in r.kv:
        kv.zero_()
    return r


@pytest.mark.parametrize("n", [1, 2])
def test_greedy_generation_graph_matches_eager_and_oracle(n):
    """Two prompts of 24 and 9 tokens on a 2-layer 0.6B-shaped model: the graph
    replay and the eager loop give identical ids and logits; each id equals the
    oracle's until a step whose top-2 logit margin is within MARGIN (there both
    ids are correct and the sequences may part); the last logits match where no
    sequence parted."""
    s = synth.QWEN3_06B
    prompts = _prompts(s.vocab, (24, 9), seed=7 + n)
    cap = 64
    r = _runner(s, n, len(prompts), cap, sum(len(p) for p in prompts))
    ids_graph, logits_graph = r.generate(prompts, STEPS, graph=True)
    logits_graph = logits_graph.clone()
    ids_eager, logits_eager = r.generate(prompts, STEPS, graph=False)
    assert ids_graph == ids_eager
    assert torch.equal(logits_graph, logits_eager)

    shape = oi.shape_of(s, num_layers=LAYERS)
    lw = [oi.layer_weights(s, li, perturbed_norms=True) for li in range(LAYERS)]
    hw = oi.head_weights(s, perturbed_norms=True)
    for b, p in enumerate(prompts):
        tokens, margins, last = of.greedy_generate(torch.tensor(p), lw, hw, shape, STEPS, kv_dtype=KV_DTYPE)
        parted = False
        for k in range(STEPS):
            if ids_graph[b][k] != tokens[k]:
                assert margins[k] <= MARGIN, (
                    f"seq {b} step {k}: id {ids_graph[b][k]} != oracle {tokens[k]} at margin {margins[k]:.3f}")
                parted = True
                break
        if not parted:
            assert_close(logits_graph[b].cpu(), last, f"last logits of seq {b}")
