"""tp_lm_head_argmax_static: the LM-head + argmax call for callers that cannot
allocate device memory (no workspace; its scratch is a fixed array inside the
library).  Checked through the C ABI against tp_lm_head_argmax on the same
inputs, on two calls in a row (the second call reuses the array the first one
left behind), against the oracle's logits and greedy ids, and with ids only
(no logits).  Kept in a file of its own that runs after the other tests."""

import numpy as np
import pytest
import torch

import synth
import synth.device as sd
from oracle import forward as of
from oracle import inputs as oi
from tests.gpu_harness import MARGIN, TOL, assert_close, model_config, oracle_head

pytestmark = pytest.mark.gpu


def _batch_inputs(q_lens, seed_stream):
    from tensor_transformer_forward_gb300 import Batch
    ctx_lens = [0] * len(q_lens)
    batch = Batch(q_lens, ctx_lens, list(range(len(q_lens))), num_prefill=sum(1 for q in q_lens if q > 1))
    h = torch.empty(sum(q_lens), synth.QWEN3_06B.hidden, dtype=torch.bfloat16, device="cuda")
    sd.fill_normal(h, synth.SEED_ACTIVATIONS, seed_stream, 1.0)
    return batch, h.float()


def test_static_scratch_lm_head_matches_workspace_version_and_oracle_twice():
    import tensor_transformer_forward_gb300 as tpf
    s, n = synth.QWEN3_06B, 2
    ctx = tpf.Context(model_config(s, n))
    head = ctx.alloc_head_shards()
    tpf.tp_shard_weights(ctx, head, head=sd.head_weights(s))
    ctx.init_workspace(64, 16, 64)  # only the existing entry point uses it
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    hw = oracle_head(s, False)
    shape = oi.shape_of(s)
    for call, (q_lens, stream) in enumerate((([3, 1, 1, 7, 1], 101), ([1] * 9 + [12], 102))):
        batch, hidden = _batch_inputs(q_lens, stream)
        B = len(q_lens)
        ref_ids = torch.full((B,), -1, dtype=torch.int32, device="cuda")
        ref_logits = torch.empty(B, s.vocab, dtype=torch.float32, device="cuda")
        tpf.tp_lm_head_argmax(ctx, head, batch, hidden, ref_ids, status, ref_logits)
        ids = torch.full((B,), -1, dtype=torch.int32, device="cuda")
        logits = torch.empty(B, s.vocab, dtype=torch.float32, device="cuda")
        tpf.binding.tp_lm_head_argmax_static(ctx, head, batch, hidden, ids, status, logits)
        ids_only = torch.full((B,), -1, dtype=torch.int32, device="cuda")
        tpf.binding.tp_lm_head_argmax_static(ctx, head, batch, hidden, ids_only, status)
        torch.cuda.synchronize()
        assert tpf.tp_read_status(status) == tpf.TP_OK
        assert torch.equal(ids.cpu(), ref_ids.cpu()), f"call {call}: ids differ"
        assert torch.equal(ids_only.cpu(), ref_ids.cpu()), f"call {call}: ids-only call differs"
        for b in range(B):
            assert_close(logits[b].cpu(), ref_logits[b].double().cpu(), f"call {call} logits of seq {b}", TOL)
        # the ids are the argmax of the logits each call produced
        assert torch.equal(ids.long().cpu(), torch.argmax(logits, dim=-1).cpu())
        # against the oracle: the last row of each sequence (the same bf16 values as
        # the device's hidden rows), final norm, all of the vocabulary
        cu = np.concatenate([[0], np.cumsum(q_lens)])
        last = hidden[torch.as_tensor(cu[1:] - 1, device="cuda")].double().cpu()
        ref = of.lm_head(last, hw, shape)
        for b in range(B):
            assert_close(logits[b].cpu(), ref[b], f"call {call} logits of seq {b} vs oracle", TOL)
            top2 = torch.topk(ref[b], 2).values
            if float(top2[0] - top2[1]) > MARGIN:
                assert int(ids[b]) == int(torch.argmax(ref[b])), f"call {call}: greedy id of seq {b}"


def test_static_scratch_rejects_sizes_beyond_its_limit():
    import tensor_transformer_forward_gb300 as tpf
    s = synth.QWEN3_06B
    ctx = tpf.Context(model_config(s, 1))
    head = ctx.alloc_head_shards()
    tpf.tp_shard_weights(ctx, head, head=sd.head_weights(s))
    batch, hidden = _batch_inputs([1] * 65, 103)
    ids = torch.empty(65, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(tpf.TPError) as e:
        tpf.binding.tp_lm_head_argmax_static(ctx, head, batch, hidden, ids, status)
    assert e.value.status == tpf.TP_ERR_INVALID_ARG
