"""Parity at the workloads' full sizes, in the launch configuration the
benchmark times: every sequence of the single-layer prefill checked element by
element; for the large decode and full-model batches, sampled sequences (each
sequence is independent, so the oracle computes just those)."""

import pytest

import synth
from tests.gpu_harness import GpuStep, check_step

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n", [1, 2])
def test_qwen3_06b_layer_prefill_2048(n):
    w = synth.WORKLOADS["qwen3_0.6b_layer_prefill2048"]
    g = GpuStep(w, n, head=False)
    check_step(g, [0], head=False)


@pytest.mark.parametrize("n", [1, 2, 4])
def test_qwen3_06b_layer_decode_64x4096_with_head(n):
    w = synth.WORKLOADS["qwen3_0.6b_layer_decode64x4096"]
    g = GpuStep(w, n)
    check_step(g, [0, 31, 63])


def test_qwen3_32b_layer_tp16_decode_32x2048_with_untied_head():
    """32B layer at tp 16 (each kv head replicated on two ranks) and the untied
    151936 x 5120 vocab-parallel LM head (16 slices of 9496 rows)."""
    w = synth.WORKLOADS["qwen3_32b_layer_tp16_decode32x2048"]
    g = GpuStep(w, 16)
    check_step(g, [0, 17, 31])


def test_qwen3_32b_layer_tp16_prefill_1024_with_untied_head():
    w = synth.WORKLOADS["qwen3_32b_layer_tp16_prefill1024"]
    g = GpuStep(w, 16)
    check_step(g, [0])


@pytest.mark.parametrize("n", [1, 2, 4])
def test_qwen3_06b_model_mixed_step(n):
    """28 layers, 4 x 512 prefill + 128 decode at ctx 2048, from ids, greedy ids."""
    w = synth.WORKLOADS["qwen3_0.6b_model_mixed"]
    g = GpuStep(w, n)
    check_step(g, [0, 4, 131])
    assert g.runner.ctx.rank_sum_count() == 2 * 28 + 1


@pytest.mark.parametrize("workload,seqs", [("qwen3_0.6b_layer_prefill2048", [0]),
                                           ("qwen3_0.6b_layer_decode64x4096", [0, 31, 63])])
def test_greedy_ids_from_the_last_fp16_rows(workload, seqs):
    """Without logits the LM head reads the last tokens' fp16 rows that the down_proj
    epilogue left (one sequence, or one token per sequence): the final norm's weight
    is folded into the head and its positive row scale cannot move the argmax."""
    w = synth.WORKLOADS[workload]
    g = GpuStep(w, 2, logits=False)
    check_step(g, seqs)
