"""Paged KV cache (zero-to-sglang "Chapter 9", section 3.3: the engine sets up the
KV cache and its page table) on the GPU: each sequence's positions live in pages
of 128 or 256 positions drawn as a shuffled, non-contiguous set, found through a
page table in the batch.  Parity with the oracle (whose cache is a plain tensor
per sequence), bit-for-bit equality with the contiguous cache on the same inputs,
and out-of-cache page entries caught by the kernels' checks."""

import pytest
import torch

import synth
from tests.gpu_harness import GpuStep, check_step

pytestmark = pytest.mark.gpu

S06 = synth.QWEN3_06B


def _same_outputs(a: GpuStep, b: GpuStep, seqs):
    assert torch.equal(a.hidden, b.hidden), "residual stream differs between paged and contiguous caches"
    if a.logits is not None:
        assert torch.equal(a.logits, b.logits)
    assert torch.equal(a.out_ids, b.out_ids)
    for s in seqs:
        for li in range(a.L):
            c0 = a.w.ctx_lens[s]
            p1 = c0 + a.w.q_lens[s]
            assert torch.equal(a.runner.kv_positions(li, s, 0, p1), b.runner.kv_positions(li, s, 0, p1))


@pytest.mark.parametrize("page_size,n", [(128, 2), (256, 1), (128, 4)])
def test_paged_mixed_batch_matches_oracle_and_contiguous(page_size, n):
    """Two layers from ids: prefill sequences with and without cached context
    (lengths that cross page boundaries, ragged against the 128-key tiles) and
    decode sequences from 0 to 900 cached positions, then the vocab head."""
    w = synth.Workload("paged_mixed", S06, (n,), ((300, 0), (70, 130), (129, 127)), (0, 127, 128, 129, 900, 5),
                       2, True)
    g = GpuStep(w, n, page_size=page_size)
    assert g.runner.page_table is not None
    rows = g.runner.page_table
    assert not all(bool((rows[b, 1:] == rows[b, :-1] + 1).all()) for b in range(rows.shape[0])), "pages contiguous"
    check_step(g, list(range(w.num_seqs)))
    c = GpuStep(w, n)
    _same_outputs(g, c, range(w.num_seqs))


def test_paged_32b_layer_tp16_replicated_kv():
    """32B-shaped layer at tp 16 (each kv head replicated on two ranks): the
    replicas of a page are written by both holding ranks and read by their own."""
    w = synth.Workload("paged_tp16", synth.QWEN3_32B, (16,), ((200, 0),), (33, 300, 255), 1, False)
    g = GpuStep(w, 16, head=False, page_size=128)
    check_step(g, [0, 1, 2, 3], head=False)
    c = GpuStep(w, 16, head=False)
    _same_outputs(g, c, range(w.num_seqs))


def test_paged_decode_64_sequences_long_context():
    """The 0.6B decode workload's shape (64 sequences, 4096 cached positions) on a
    paged cache of 128-position pages: 33 pages per sequence, split key ranges."""
    w = synth.WORKLOADS["qwen3_0.6b_layer_decode64x4096"]
    g = GpuStep(w, 2, page_size=128)
    check_step(g, [0, 31, 63])
    c = GpuStep(w, 2)
    assert torch.equal(g.hidden, c.hidden) and torch.equal(g.out_ids, c.out_ids)


def test_page_entries_outside_the_cache_flag_bad_token():
    """A page table entry beyond the cache's pages (or negative), on a position the
    step writes or reads, is caught by the kernels' own checks: nothing outside the
    cache is touched and the status word reports TP_ERR_BAD_TOKEN."""
    from tensor_transformer_forward_gb300 import TP_ERR_BAD_TOKEN, TP_OK, Batch, tp_read_status
    from tensor_transformer_forward_gb300.runner import TPRunner
    from tests.gpu_harness import model_config
    import synth.device as sd
    s = synth.TINY
    r = TPRunner(model_config(s, 2), 1, max_seqs=2, capacity=256, max_tokens=16, page_size=128)
    r.load_layer(0, sd.layer_weights(s, 0))
    hidden = torch.randn(8, s.hidden, device="cuda")
    good = r.page_table.clone()
    cases = []
    t = good.clone()
    t[1, 1] = r.num_pages            # decode sequence at position 200 reads page 1 of its row
    cases.append(([1, 1], [3, 200], t, 0))
    t = good.clone()
    t[0, 0] = -1                     # prefill sequence's first page
    cases.append(([5, 1], [0, 4], t, 1))
    for q, c, table, npre in cases:
        r.status.zero_()
        b = Batch(q, c, None, npre, page_table=table, page_size=128)
        h = hidden[: b.num_tokens].clone()
        r.layer(0, b, h)
        assert tp_read_status(r.status) == TP_ERR_BAD_TOKEN
    r.status.zero_()
    b = Batch([1, 1], [3, 200], None, 0, page_table=good, page_size=128)
    r.layer(0, b, hidden[:2].clone())
    assert tp_read_status(r.status) == TP_OK
