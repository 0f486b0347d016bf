"""Whole-step parity on the GPU against the fp64 oracle at sizes the oracle
finishes in seconds: prefill, decode, mixed batches, several layers, the
vocab head with argmax, every tp size the shapes allow (incl. KV-head
replication).  Tolerance: max |err| <= 2e-2 x RMS(reference) per tensor;
greedy ids equal where the reference top-2 margin exceeds 0.05."""

import pytest

import synth
from oracle import forward as of
from tests.gpu_harness import MARGIN, GpuStep, assert_close, check_step, oracle_run_sp

pytestmark = pytest.mark.gpu

S06 = synth.QWEN3_06B


@pytest.mark.parametrize("n", [1, 2, 4])
def test_tiny_workload_from_ids(n):
    """The tiny workload: hidden 256, 4 q / 2 kv heads, 8 prefill tokens from ids,
    one layer and the vocab head (n=4 replicates each kv head on 2 ranks)."""
    w = synth.WORKLOADS["tiny_prefill8"]
    g = GpuStep(w, n, perturbed=True)
    check_step(g, [0])
    assert g.runner.ctx.rank_sum_count() == 2 * 1 + 1


@pytest.mark.parametrize("n", [1, 2, 4])
def test_decode_varied_context_lengths(n):
    """Decode: one new token for sequences with 0 .. 2047 cached positions
    (several key splits, ragged tails), then the LM head."""
    ctxs = (0, 1, 63, 64, 513, 1000, 2047, 77)
    w = synth.Workload("decode_var", S06, (n,), (), ctxs, 1, False)
    g = GpuStep(w, n)
    check_step(g, list(range(len(ctxs))))


def test_decode_thin_last_wave_split_further():
    """40 decode sequences at tp 2 (320 (sequence, rank, kv head) units): on a GPU
    holding 304 resident decode CTAs the last 16 units form a thin last wave and
    take 4 key splits each.  Those units belong to the last two sequences: one with
    a single key (three empty splits) and one with 2200; the others ragged."""
    ctxs = tuple((i * 613) % 2300 for i in range(38)) + (0, 2200)
    w = synth.Workload("decode_tail", S06, (2,), (), ctxs, 1, False)
    g = GpuStep(w, 2)
    check_step(g, [0, 1, 17, 37, 38, 39])


def test_decode_persistent_ctas_take_many_items():
    """200 decode sequences at tp 2 (1600 (sequence, rank, kv head) units) over
    two layers: each resident decode CTA takes several items in turn, whole units
    first and key splits of the last units (80 left after five rounds of 304,
    three splits each); ragged lengths with a one-key context among the split
    ones.  The second layer's launch draws from the ticket counter the first one
    reset."""
    ctxs = tuple((i * 397) % 900 for i in range(198)) + (0, 1500)
    w = synth.Workload("decode_many", S06, (2,), (), ctxs, 2, False)
    g = GpuStep(w, 2, head=False)
    check_step(g, [0, 1, 57, 120, 189, 190, 197, 198, 199], head=False)


@pytest.mark.parametrize("n", [1, 2])
def test_prefill_with_cache_offset_and_ragged_lengths(n):
    """Prefill sequences with cached context (mask tril(S - T)) and lengths that
    are not multiples of the 64/128 tiles."""
    w = synth.Workload("prefill_ctx", S06, (n,), ((130, 0), (70, 50), (1, 9), (65, 200)), (), 1, False)
    g = GpuStep(w, n, perturbed=True)
    check_step(g, [0, 1, 2, 3])


def test_mixed_batch_two_layers_from_ids():
    """Mixed step: two prefill sequences and five decode sequences, embedding
    from ids, two layers, the vocab head."""
    w = synth.Workload("mixed_small", S06, (2,), ((130, 0), (70, 0)), (5, 100, 300, 1, 700), 2, True)
    g = GpuStep(w, 2)
    check_step(g, list(range(7)))
    assert g.runner.ctx.rank_sum_count() == 2 * 2 + 1


def test_32b_layer_tp16_replicated_kv():
    """32B-shaped layer at tp 16: 4 q heads and one replicated kv head per rank;
    a prefill sequence and decode sequences (layer only: the untied 32B vocab
    head is checked at the 0.6B shape)."""
    w = synth.Workload("tp16_small", synth.QWEN3_32B, (16,), ((40, 0),), (33, 200), 1, False)
    g = GpuStep(w, 16, head=False)
    check_step(g, [0, 1, 2], head=False)


@pytest.mark.parametrize("n", [1, 2, 4])
def test_long_k_residual_gemm_split_in_two(n):
    """down_proj with 256 K blocks (intermediate 16384) over 1297 tokens (24 tiles
    of 256 x 256).  At tp 1 and 2 (one or two rank segments) o_proj and down_proj
    run on 4-CTA clusters whose two CTA pairs take one K half each and exchange
    their partials through distributed shared memory; at tp 4 down_proj runs on
    CTA pairs with the rank segments split in two halves that meet in split-K
    partials in global memory.  The residual they leave against the oracle."""
    s = synth.ModelShape(hidden=1024, num_q_heads=8, num_kv_heads=4, head_dim=128, intermediate=16384, vocab=1000,
                         num_layers=1)
    w = synth.Workload("long_k_resid", s, (n,), ((1280, 0),), (17,), 1, True)
    g = GpuStep(w, n)
    check_step(g, [0, 1])


@pytest.mark.parametrize("nseq", [150, 180, 256])
def test_head_many_sequences_token_tiles(nseq):
    """The vocab head for 129..256 sequences streams the weights once against one
    token tile of 160, 192 or 256 columns (the rows past the last sequence are
    zero fill and never read back); ids and logits of sampled sequences."""
    w = synth.Workload("head_many", S06, (2,), (), tuple((i * 37) % 200 for i in range(nseq)), 1, True)
    g = GpuStep(w, 2)
    check_step(g, [0, nseq // 2, nseq - 1])


def test_untied_head_uneven_vocab():
    """Untied LM head with a vocab that leaves the last rank a shorter slice
    (padded columns must never win the argmax)."""
    s = synth.ModelShape(hidden=256, num_q_heads=6, num_kv_heads=3, head_dim=64, intermediate=384, vocab=1001,
                         num_layers=1, tie_word_embeddings=False)
    w = synth.Workload("untied_uneven", s, (3,), ((17, 0),), (5, 9), 1, True)
    g = GpuStep(w, 3, perturbed=True)
    check_step(g, [0, 1, 2])


def test_slot_or_length_outside_the_cache_flags_bad_token():
    """A batch whose device arrays point outside the cache (a slot >= max_seqs,
    or a cached length beyond the capacity) is caught by the kernels' own bounds
    checks: nothing outside the cache is read or written and the status word
    reports TP_ERR_BAD_TOKEN."""
    import torch
    import synth.device as sd
    from tensor_transformer_forward_gb300 import TP_ERR_BAD_TOKEN, TP_OK, tp_read_status
    from tensor_transformer_forward_gb300.runner import TPRunner
    from tests.gpu_harness import model_config
    s = synth.TINY
    r = TPRunner(model_config(s, 2), 1, max_seqs=2, capacity=64, max_tokens=16)
    r.load_layer(0, sd.layer_weights(s, 0))
    hidden = torch.randn(8, s.hidden, device="cuda")
    cases = [r.make_batch([1, 1], [3, 4], [0, 2]),            # decode, slot 2 of 2
             r.make_batch([5, 1], [0, 4], [3, 0]),            # prefill, slot 3 of 2
             r.make_batch([1, 1], [3, 4], [0, 1])]            # decode, length tampered below
    cases[2].ctx_len[1] = 100                                 # 101 keys in a 64-position cache
    for batch in cases:
        r.status.zero_()
        h = hidden[: batch.num_tokens].clone()
        r.layer(0, batch, h)
        assert tp_read_status(r.status) == TP_ERR_BAD_TOKEN
    r.status.zero_()
    ok = r.make_batch([1, 1], [3, 4], [0, 1])
    r.layer(0, ok, hidden[:2].clone())
    assert tp_read_status(r.status) == TP_OK


def test_decode_large_weights_64dim_heads_few_tokens():
    """Few tokens against large weights take the weights-on-M tiles (128 features x
    the tokens): 64-dim heads (two per tile), a prefill sequence among decode
    sequences, K split over CTAs, tp 2."""
    s = synth.ModelShape(hidden=4096, num_q_heads=32, num_kv_heads=8, head_dim=64, intermediate=11008, vocab=2048,
                         num_layers=1, tie_word_embeddings=False)
    w = synth.Workload("large_w_decode", s, (2,), ((9, 0),), (3, 70, 200, 0), 1, False)
    g = GpuStep(w, 2, perturbed=True)
    check_step(g, list(range(5)))


@pytest.mark.parametrize("q_heads,kv_heads", [(16, 2), (8, 8)])
def test_decode_query_groups_of_eight_and_one(q_heads, kv_heads):
    """The tensor-core decode attention with 8 query heads per kv head at tp 2 (the
    smallest rings: two 16 KB slots each for K and V) and with one (multi-head
    attention); ragged contexts (one key, a partial last tile, 2200 keys) and a
    prefill sequence beside them."""
    s = synth.ModelShape(hidden=512, num_q_heads=q_heads, num_kv_heads=kv_heads, head_dim=128, intermediate=768,
                         vocab=1000, num_layers=1)
    w = synth.Workload("decode_groups", s, (2,), ((40, 0),), (0, 130, 2200, 511, 77), 1, False)
    g = GpuStep(w, 2)
    check_step(g, list(range(6)))


@pytest.mark.parametrize("prefill,decode", [(((130, 0),), (3, 70)), (((9, 0),), (3, 70, 200))])
def test_hidden_not_a_multiple_of_128(prefill, decode):
    """hidden 4160 = 32.5 x 128: the residual epilogues' last feature tile lies half
    outside the rows (token tiles for the 132-token step, weights-on-M rows for the
    12-token one), the embedding's last chunk round is partial, and the deferred
    norms add 130 column groups per row."""
    s = synth.ModelShape(hidden=4160, num_q_heads=32, num_kv_heads=8, head_dim=64, intermediate=11008, vocab=2048,
                         num_layers=1, tie_word_embeddings=False)
    w = synth.Workload("ragged_hidden", s, (2,), prefill, decode, 1, True)
    g = GpuStep(w, 2, perturbed=True)
    check_step(g, list(range(w.num_seqs)))


@pytest.mark.parametrize("n", [2, 4])
def test_sequence_parallel_token_chunks(n):
    """Sequence parallelism ("Tensor parallelism from scratch", Exercises, 1): one
    prefill sequence of 301 tokens from ids, two layers and the head.  On one GPU
    the reduce-scatter's token chunks are contiguous row ranges of the rank-summed
    [T, H] residual that the row GEMM epilogues write, and the all-gather before a
    column GEMM is the identity on that layout: rows token_chunk(T, n, r) of the
    device's residual are rank r's chunk of the oracle's sequence-parallel form."""
    T = 301
    w = synth.Workload("sp_prefill", S06, (n,), ((T, 0),), (), 2, True)
    g = GpuStep(w, n)
    sp = oracle_run_sp(w, 0, 2, n)
    for r in range(n):
        a, b = of.token_chunk(T, n, r)
        assert_close(g.hidden[a:b].float().cpu(), sp.hidden_chunks[r], f"token chunk of rank {r}")
    assert_close(g.logits[0].cpu(), sp.logits, "logits")
    top2 = sp.logits.topk(2).values
    if float(top2[0] - top2[1]) > MARGIN:
        assert int(g.out_ids[0]) == sp.next_id


@pytest.mark.parametrize("prefill", [True, False])
def test_fp16_saturation_is_reported(prefill):
    """GEMM operands are fp16 and clamp at +-65504: residual rows scaled by 2^17
    (a host-side input, no fault) must set TP_ERR_SATURATED in the status word,
    and so must a weight outside the fp16 range at shard time; the same inputs at
    their normal scale leave the word clear."""
    import torch
    import synth.device as sd
    from tensor_transformer_forward_gb300 import TP_ERR_SATURATED, TP_OK, tp_read_status, tp_shard_weights
    from tensor_transformer_forward_gb300.runner import TPRunner
    from tests.gpu_harness import model_config
    s = synth.QWEN3_06B
    r = TPRunner(model_config(s, 2), 1, max_seqs=4, capacity=128, max_tokens=64)
    full = sd.layer_weights(s, 0)
    r.load_layer(0, full)
    q = [48, 1, 1, 1] if prefill else [1, 1, 1, 1]
    batch = r.make_batch(q, [0, 5, 9, 17], [0, 1, 2, 3], num_prefill=1 if prefill else 0)
    h = torch.empty(batch.num_tokens, s.hidden, dtype=torch.bfloat16, device="cuda")
    sd.fill_normal(h, synth.SEED_ACTIVATIONS, 7, 1.0)
    r.status.zero_()
    r.step(batch, hidden=h.float(), run_head=False)
    assert tp_read_status(r.status) == TP_OK
    r.step(batch, hidden=h.float() * 2.0 ** 17, run_head=False)
    assert tp_read_status(r.status) == TP_ERR_SATURATED
    # a weight beyond the fp16 range: flagged when the shards are made
    big = {k: v.clone() for k, v in full.items()}
    big["down"][3, 5] = 1.0e5
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    tp_shard_weights(r.ctx, r.ctx.alloc_layer_shards(), layer=big, status=st)
    assert tp_read_status(st) == TP_ERR_SATURATED
    st.zero_()
    tp_shard_weights(r.ctx, r.ctx.alloc_layer_shards(), layer=full, status=st)
    assert tp_read_status(st) == TP_OK
