"""Property tests of the oracle's sharded forms (CPU): over random shapes that the
shard rules of "Tensor parallelism from scratch" allow (kv-head replication, uneven
vocab slices, tied or untied heads), random tp sizes, token counts and cached
lengths, the all-reduce TP emulation and the sequence-parallel form both equal the
unsharded forward, which is itself pinned against brute force.

The cases come from a seeded generator of their own (always run), and, where the
``hypothesis`` package is installed, also from its search."""

import random

import pytest
import torch

from oracle import forward as of

try:
    import hypothesis
    st = hypothesis.strategies
except ImportError:  # the seeded cases below still run
    hypothesis = None

D = torch.float64


def _case(pick, assume):
    """One case from a chooser pick(kind, options) and a rejection hook assume(cond)."""
    nkv = pick("choice", [1, 2, 4])
    group = pick("choice", [1, 2, 4])
    nq = nkv * group
    n = pick("choice", [d for d in (1, 2, 4, 8) if nq % d == 0])
    hd = pick("choice", [8, 12, 16])
    hidden = pick("choice", [16, 32, 48])
    inter = n * pick("int", (1, 6)) * 4
    vocab = pick("int", (2 * n + 1, 97))
    tied = pick("choice", [False, True])
    shape = of.Shape(hidden=hidden, num_q_heads=nq, num_kv_heads=nkv, head_dim=hd, intermediate=inter,
                     vocab=vocab, num_layers=2, tie_word_embeddings=tied)
    try:
        of.validate_tp(shape, n)
    except of.ShardError:
        assume(False)
        return None
    T = pick("int", (1, 9))
    ctx = pick("int", (0, 6))
    seed = pick("int", (0, 2**31 - 1))
    return shape, n, T, ctx, seed


def _seeded_cases(count: int, seed: int = 20251202):
    rng = random.Random(seed)

    def pick(kind, opts):
        return rng.choice(opts) if kind == "choice" else rng.randint(*opts)

    out = []
    while len(out) < count:
        c = _case(pick, lambda ok: None)
        if c is not None:
            out.append(c)
    return out


def _inputs(shape, T, ctx, seed):
    g = torch.Generator().manual_seed(seed)
    H, nq, nkv, hd, I = shape.hidden, shape.num_q_heads, shape.num_kv_heads, shape.head_dim, shape.intermediate
    r = lambda *s: torch.randn(*s, dtype=D, generator=g) * 0.2  # noqa: E731
    layers = [of.LayerWeights(q=r(nq * hd, H), k=r(nkv * hd, H), v=r(nkv * hd, H), o=r(H, nq * hd),
                              gate=r(I, H), up=r(I, H), down=r(H, I), in_norm=1 + r(H), post_norm=1 + r(H),
                              q_norm=1 + r(hd), k_norm=1 + r(hd)) for _ in range(2)]
    emb = torch.randn(shape.vocab, H, dtype=D, generator=g)
    lm = emb if shape.tie_word_embeddings else torch.randn(shape.vocab, H, dtype=D, generator=g)
    hw = of.HeadWeights(embed=emb, lm_head=lm, final_norm=1 + r(H))
    kc = [torch.randn(nkv, ctx, hd, dtype=D, generator=g) for _ in range(2)]
    vc = [torch.randn(nkv, ctx, hd, dtype=D, generator=g) for _ in range(2)]
    seq = of.SeqInput(hidden=None, ids=torch.randint(0, shape.vocab, (T,), generator=g), k_cache=kc, v_cache=vc)
    return layers, hw, seq


def _close(a, b):
    scale = max(float(b.abs().max()), 1.0)
    return a.shape == b.shape and float((a - b).abs().max()) <= 1e-11 * scale


def _check(case):
    shape, n, T, ctx, seed = case
    layers, hw, seq = _inputs(shape, T, ctx, seed)
    ref = of.run_sequence(seq, layers, hw, shape, n=0)
    comm = of.Comm()
    tp = of.run_sequence(seq, layers, hw, shape, n=n, comm=comm)
    sp = of.run_sequence_sp(seq, layers, hw, shape, n)
    assert comm.num_all_reduce == 2 * len(layers) + 1
    for got in (tp.hidden, torch.cat(sp.hidden_chunks)):
        assert _close(got, ref.hidden)
    for got in (tp.logits, sp.logits):
        assert _close(got, ref.logits)
    assert tp.next_id == ref.next_id == sp.next_id
    for a, b in zip(tp.k_cache + tp.v_cache + sp.k_cache + sp.v_cache, 2 * (ref.k_cache + ref.v_cache)):
        assert _close(a, b)


SEEDED = _seeded_cases(40)


@pytest.mark.parametrize("case", SEEDED, ids=[f"n{c[1]}-nq{c[0].num_q_heads}-nkv{c[0].num_kv_heads}-T{c[2]}-ctx{c[3]}"
                                              for c in SEEDED])
def test_sharded_forms_equal_the_unsharded_forward_seeded(case):
    _check(case)


def test_seeded_cases_cover_replication_uneven_vocab_and_both_head_kinds():
    assert any(c[0].num_kv_heads < c[1] for c in SEEDED)           # kv heads replicated
    assert any(c[0].vocab % c[1] for c in SEEDED)                   # uneven vocab slices
    assert {c[0].tie_word_embeddings for c in SEEDED} == {False, True}
    assert {c[1] for c in SEEDED} >= {1, 2, 4}


if hypothesis is not None:
    @st.composite
    def cases(draw):
        def pick(kind, opts):
            return draw(st.sampled_from(opts)) if kind == "choice" else draw(st.integers(*opts))
        return _case(pick, hypothesis.assume)

    @hypothesis.settings(max_examples=40, deadline=None, derandomize=True)
    @hypothesis.given(cases())
    def test_sharded_forms_equal_the_unsharded_forward(case):
        _check(case)
