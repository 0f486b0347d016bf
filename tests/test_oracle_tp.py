"""Pins of the oracle's tensor-parallel emulation: the invariant sharded ==
unsharded, the collective count, the shard rules and the numbers printed in
"Tensor parallelism from scratch" (tests/golden/)."""

import json
import os

import numpy as np
import pytest
import torch

from oracle import forward as of

D = torch.float64
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _weights(shape, seed, layers=1):
    g = torch.Generator().manual_seed(seed)
    H, nq, nkv, hd, I = shape.hidden, shape.num_q_heads, shape.num_kv_heads, shape.head_dim, shape.intermediate
    r = lambda *s: torch.randn(*s, dtype=D, generator=g) * 0.2  # noqa: E731
    ls = [of.LayerWeights(q=r(nq * hd, H), k=r(nkv * hd, H), v=r(nkv * hd, H), o=r(H, nq * hd),
                          gate=r(I, H), up=r(I, H), down=r(H, I), in_norm=1 + r(H), post_norm=1 + r(H),
                          q_norm=1 + r(hd), k_norm=1 + r(hd)) for _ in range(layers)]
    emb = torch.randn(shape.vocab, H, dtype=D, generator=g)
    lm = emb if shape.tie_word_embeddings else torch.randn(shape.vocab, H, dtype=D, generator=g)
    return ls, of.HeadWeights(embed=emb, lm_head=lm, final_norm=1 + r(H))


def _seq(shape, seed, T, ctx, layers, ids=True):
    g = torch.Generator().manual_seed(seed)
    kc = [torch.randn(shape.num_kv_heads, ctx, shape.head_dim, dtype=D, generator=g) for _ in range(layers)]
    vc = [torch.randn(shape.num_kv_heads, ctx, shape.head_dim, dtype=D, generator=g) for _ in range(layers)]
    if ids:
        return of.SeqInput(hidden=None, ids=torch.randint(0, shape.vocab, (T,), generator=g), k_cache=kc, v_cache=vc)
    return of.SeqInput(hidden=torch.randn(T, shape.hidden, dtype=D, generator=g), ids=None, k_cache=kc, v_cache=vc)


SMALL = of.Shape(hidden=64, num_q_heads=8, num_kv_heads=4, head_dim=16, intermediate=96, vocab=103,
                 num_layers=2, tie_word_embeddings=False)


@pytest.mark.parametrize("n", [1, 2, 4, 8])
def test_tp_equals_unsharded(n):
    """Invariant of the method: the sharded result equals the single-process one
    up to summation order (n=8 > 4 kv heads exercises replication)."""
    layers, hw = _weights(SMALL, 10, layers=2)
    seq = _seq(SMALL, 11, T=5, ctx=3, layers=2)
    ref = of.run_sequence(seq, layers, hw, SMALL, n=0)
    comm = of.Comm()
    got = of.run_sequence(seq, layers, hw, SMALL, n=n, comm=comm)
    assert torch.allclose(got.hidden, ref.hidden, rtol=1e-12, atol=1e-12)
    assert torch.allclose(got.logits, ref.logits, rtol=1e-12, atol=1e-11)
    assert got.next_id == ref.next_id
    for a, b in zip(got.k_cache + got.v_cache, ref.k_cache + ref.v_cache):
        assert torch.allclose(a, b, rtol=1e-12, atol=1e-12)
    # one sum for the embedding + two per layer, one gather for the logits
    assert comm.num_all_reduce == 2 * 2 + 1 and comm.num_all_gather == 1


def test_rank_sum_count_57_for_28_layers():
    shape = of.Shape(hidden=32, num_q_heads=4, num_kv_heads=2, head_dim=8, intermediate=32, vocab=40,
                     num_layers=28)
    layers, hw = _weights(shape, 12, layers=28)
    seq = _seq(shape, 13, T=4, ctx=0, layers=28)
    comm = of.Comm()
    got = of.run_sequence(seq, layers, hw, shape, n=2, comm=comm)
    gold = json.load(open(os.path.join(GOLDEN, "tp_qwen3_0.6b_tp2.json")))
    assert comm.num_all_reduce == gold["all_reduce_per_prefill_forward"] == 57
    ref = of.run_sequence(seq, layers, hw, shape, n=0)
    assert got.next_id == ref.next_id


def test_fp32_error_is_summation_order_sized():
    """In fp32 the TP-vs-single logits error is of the order the page prints
    (1.4e-5, attributed to summation order); in fp64 it vanishes."""
    layers, hw = _weights(SMALL, 14, layers=2)
    seq = _seq(SMALL, 15, T=6, ctx=0, layers=2)
    f32 = lambda t: t.to(torch.float32)  # noqa: E731
    l32 = [of.LayerWeights(**{k: f32(v) for k, v in vars(w).items()}) for w in layers]
    h32 = of.HeadWeights(embed=f32(hw.embed), lm_head=f32(hw.lm_head), final_norm=f32(hw.final_norm))
    s32 = of.SeqInput(hidden=None, ids=seq.ids, k_cache=[f32(k) for k in seq.k_cache],
                      v_cache=[f32(v) for v in seq.v_cache])
    e32 = (of.run_sequence(s32, l32, h32, SMALL, n=2).logits - of.run_sequence(s32, l32, h32, SMALL, n=0).logits)
    e64 = (of.run_sequence(seq, layers, hw, SMALL, n=2).logits - of.run_sequence(seq, layers, hw, SMALL, n=0).logits)
    assert 0 < float(e32.abs().max()) < 1e-4
    assert float(e64.abs().max()) < 1e-12


def test_parameter_counts_and_kv_heads_match_printed_run():
    gold = json.load(open(os.path.join(GOLDEN, "tp_qwen3_0.6b_tp2.json")))
    m = gold["model"]
    shape = of.Shape(hidden=m["hidden"], num_q_heads=m["num_q_heads"], num_kv_heads=m["num_kv_heads"],
                     head_dim=m["head_dim"], intermediate=m["intermediate"], vocab=m["vocab"],
                     num_layers=m["num_layers"], tie_word_embeddings=m["tie_word_embeddings"])
    n = gold["tp_size"]
    per_rank = [of.param_count(shape, n, r) for r in range(n)]
    full = of.param_count(shape, 1, 0)
    assert round(per_rank[0] / 1e6) == gold["params_per_rank_millions_rounded"]
    assert round(full / 1e6) == gold["params_full_millions_rounded"]
    assert per_rank[0] == per_rank[1]
    assert len(of.kv_heads_of_rank(shape, n, 0)) == gold["kv_heads_per_rank"]


def test_head_count_rules_from_page():
    gold = json.load(open(os.path.join(GOLDEN, "tp_head_count_rules.json")))
    base = dict(hidden=256, head_dim=8, intermediate=256, vocab=1024, num_layers=1)
    c0, c1, c2 = gold["cases"]
    s0 = of.Shape(num_q_heads=c0["num_q_heads"], num_kv_heads=c0["num_kv_heads"], **base)
    for n in c0["valid_tp"]:
        of.validate_tp(s0, n)
    for n in (3, 5, 6):
        with pytest.raises(of.ShardError):
            of.validate_tp(s0, n)
    s1 = of.Shape(num_q_heads=c1["num_q_heads"], num_kv_heads=c1["num_kv_heads"], **base)
    with pytest.raises(of.ShardError):
        of.validate_tp(s1, c1["tp"])
    s2 = of.Shape(num_q_heads=c2["num_q_heads"], num_kv_heads=c2["num_kv_heads"], **base)
    of.validate_tp(s2, c2["tp"])
    got = [of.kv_heads_of_rank(s2, c2["tp"], r) for r in range(c2["tp"])]
    assert got == [[g] for g in c2["kv_head_of_rank"]]


def test_uneven_splits_are_errors():
    ok = dict(hidden=64, num_q_heads=4, num_kv_heads=2, head_dim=16, intermediate=96, vocab=100, num_layers=1)
    with pytest.raises(of.ShardError):
        of.validate_tp(of.Shape(**{**ok, "intermediate": 97}), 2)
    with pytest.raises(of.ShardError):   # 3 ranks over 2 kv heads: neither a chunk nor a replica
        of.validate_tp(of.Shape(**{**ok, "num_q_heads": 6, "num_kv_heads": 2, "intermediate": 96}), 3)
    with pytest.raises(of.ShardError):   # V=5 over 4 ranks: div_ceil 2 leaves rank 3 empty
        of.validate_tp(of.Shape(**{**ok, "vocab": 5}), 4)


def test_vocab_ranges_div_ceil_and_masked_embedding():
    assert [of.vocab_range(1000, 3, r) for r in range(3)] == [(0, 334), (334, 668), (668, 1000)]
    assert [of.vocab_range(151936, 2, r) for r in range(2)] == [(0, 75968), (75968, 151936)]
    shape = of.Shape(hidden=16, num_q_heads=2, num_kv_heads=1, head_dim=8, intermediate=16, vocab=1000,
                     num_layers=0)
    g = torch.Generator().manual_seed(16)
    hw = of.HeadWeights(embed=torch.randn(1000, 16, dtype=D, generator=g), lm_head=None,
                        final_norm=torch.ones(16, dtype=D))
    hw.lm_head = hw.embed
    ids = torch.tensor([0, 333, 334, 667, 668, 999, 500])
    for n in (1, 2, 3):
        comm = of.Comm()
        assert torch.equal(of.tp_embed(ids, hw, shape, n, comm), hw.embed[ids])
        assert comm.num_all_reduce == 1
        x = torch.randn(16, dtype=D, generator=g)
        assert torch.allclose(of.tp_lm_head(x, hw, shape, n, of.Comm()), of.lm_head(x, hw, shape), atol=1e-12)


def test_shard_then_merge_layout_and_replicated_kv():
    shape = of.Shape(hidden=32, num_q_heads=8, num_kv_heads=2, head_dim=4, intermediate=64, vocab=64,
                     num_layers=1)
    (w,), _ = _weights(shape, 17)
    n = 4
    ranks = [of.shard_layer(w, shape, n, r) for r in range(n)]
    for r, rl in enumerate(ranks):
        q_rows = slice(r * 8, (r + 1) * 8)             # 2 q heads of 4 dims per rank
        g = r * 2 // 4                                 # replicated kv head
        assert torch.equal(rl.qkv[:8], w.q[q_rows])
        assert torch.equal(rl.qkv[8:12], w.k[g * 4:(g + 1) * 4])
        assert torch.equal(rl.qkv[12:16], w.v[g * 4:(g + 1) * 4])
        assert torch.equal(rl.gate_up[:16], w.gate[r * 16:(r + 1) * 16])
        assert torch.equal(rl.gate_up[16:], w.up[r * 16:(r + 1) * 16])
        assert torch.equal(rl.o, w.o[:, q_rows]) and torch.equal(rl.down, w.down[:, r * 16:(r + 1) * 16])
    # ranks 2g and 2g+1 hold bit-identical copies of kv head g
    assert torch.equal(ranks[0].qkv[8:16], ranks[1].qkv[8:16])
    assert torch.equal(ranks[2].qkv[8:16], ranks[3].qkv[8:16])
    assert not torch.equal(ranks[1].qkv[8:16], ranks[2].qkv[8:16])


def test_column_then_row_needs_no_exchange_between():
    """Between the column-split projection and the row-split one, every rank
    works only on its own slice: summing the per-rank partials of o_proj equals
    the full o_proj of the concatenated attention outputs."""
    (w,), _ = _weights(SMALL, 18)
    n = 2
    g = torch.Generator().manual_seed(19)
    attn = torch.randn(3, SMALL.num_q_heads * SMALL.head_dim, dtype=D, generator=g)
    parts = []
    for r in range(n):
        rl = of.shard_layer(w, SMALL, n, r)
        cols = of.shard_index("o", SMALL, n, r)[1]
        parts.append(attn[:, cols] @ rl.o.T)
    assert torch.allclose(of.Comm().all_reduce(parts), attn @ w.o.T, atol=1e-12)


def test_greedy_generation_cache_equals_recompute_and_tp_equals_unsharded():
    """The generation loop against two things it does not compute itself: every
    step's token and the last logits equal a cache-free forward over prompt +
    tokens so far (positions, RoPE offsets and cache appends of the loop), and the
    TP emulation generates the same tokens as the unsharded model (the page's own
    check of its 20 greedy tokens)."""
    layers, hw = _weights(SMALL, 20, layers=2)
    prompt = torch.randint(0, SMALL.vocab, (7,), generator=torch.Generator().manual_seed(21))
    tokens, margins, last = of.greedy_generate(prompt, layers, hw, SMALL, steps=6)
    assert len(tokens) == 6 and all(m >= 0 for m in margins)
    empty = [torch.zeros(SMALL.num_kv_heads, 0, SMALL.head_dim, dtype=D) for _ in layers]
    seq = prompt.clone()
    for k in range(6):
        full = of.run_sequence(of.SeqInput(None, seq, list(empty), list(empty)), layers, hw, SMALL)
        assert full.next_id == tokens[k]
        seq = torch.cat([seq, torch.tensor([tokens[k]])])
    full = of.run_sequence(of.SeqInput(None, seq, list(empty), list(empty)), layers, hw, SMALL)
    assert torch.allclose(last, full.logits, rtol=1e-10, atol=1e-10)
    tp_tokens, _, tp_last = of.greedy_generate(prompt, layers, hw, SMALL, steps=6, n=2)
    assert tp_tokens == tokens
    assert torch.allclose(tp_last, last, rtol=1e-10, atol=1e-10)
