"""Pins of the oracle's building blocks against closed forms, library routines and
brute force (no GPU).  Each check would fail on a plausible slip: a dropped
term, a wrong sign or index, a transposed operand."""

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import synth
from oracle import brute
from oracle import forward as of
from oracle import inputs as oi

D = torch.float64


def test_rms_norm_closed_forms_and_library():
    x = torch.full((5,), 3.0, dtype=D)
    w = torch.arange(1, 6, dtype=D)
    eps = 1e-6
    # constant vector c: y = c / sqrt(c^2 + eps) * w
    assert torch.allclose(of.rms_norm(x, w, eps), 3.0 / math.sqrt(9.0 + eps) * w, rtol=0, atol=1e-15)
    g = torch.Generator().manual_seed(0)
    y = torch.randn(7, 64, dtype=D, generator=g) * 4
    ones = torch.ones(64, dtype=D)
    out = of.rms_norm(y, ones, eps)
    rms = out.pow(2).mean(-1)
    assert torch.allclose(rms, y.pow(2).mean(-1) / (y.pow(2).mean(-1) + eps), rtol=1e-13)
    wv = torch.randn(64, dtype=D, generator=g)
    assert torch.allclose(of.rms_norm(y, wv, eps), F.rms_norm(y, (64,), wv, eps), rtol=1e-12, atol=1e-14)


def test_rope_identity_exact_angle_and_complex_form():
    g = torch.Generator().manual_seed(1)
    u = torch.randn(3, 6, 16, dtype=D, generator=g)
    pos0 = torch.zeros(6, dtype=torch.long)
    assert torch.equal(of.apply_rope(u, pos0, 1e6), u)
    # position 1, pair d=0 rotates by exactly 1 radian, pair d has angle theta^(-2d/hd)
    e0 = torch.zeros(1, 16, dtype=D)
    e0[0, 0] = 1.0
    r = of.apply_rope(e0, torch.tensor([1]), 1e6)
    assert abs(float(r[0, 0]) - math.cos(1.0)) < 1e-15 and abs(float(r[0, 8]) - math.sin(1.0)) < 1e-15
    # same rotation as multiplying (a + i b) by exp(i * angle) with numpy complex math
    pos = torch.tensor([0, 5, 77, 4096, 100000, 3, 9])
    v = torch.randn(7, 16, dtype=D, generator=g)
    got = of.apply_rope(v, pos, 1e6).numpy()
    a, b = v[:, :8].numpy(), v[:, 8:].numpy()
    ang = pos.numpy()[:, None].astype(np.float64) * (1e6 ** (-2.0 * np.arange(8) / 16.0))[None, :]
    z = (a + 1j * b) * np.exp(1j * ang)
    assert np.allclose(got[:, :8], z.real, atol=1e-13) and np.allclose(got[:, 8:], z.imag, atol=1e-13)


def test_rope_preserves_pairs_and_depends_on_relative_position():
    g = torch.Generator().manual_seed(2)
    q = torch.randn(1, 32, dtype=D, generator=g)
    k = torch.randn(1, 32, dtype=D, generator=g)
    dots = []
    for p in (0, 11, 2000):
        qr = of.apply_rope(q, torch.tensor([p + 7]), 1e4)
        kr = of.apply_rope(k, torch.tensor([p]), 1e4)
        dots.append(float((qr * kr).sum()))
        pair = qr[0, :16] ** 2 + qr[0, 16:] ** 2
        assert torch.allclose(pair, q[0, :16] ** 2 + q[0, 16:] ** 2, rtol=1e-12)
    assert max(dots) - min(dots) < 1e-10


def test_attention_matches_library_sdpa_with_gqa_and_offset():
    g = torch.Generator().manual_seed(3)
    nq, nkv, T, S, hd = 8, 2, 5, 12, 16
    q = torch.randn(nq, T, hd, dtype=D, generator=g)
    k = torch.randn(nkv, S, hd, dtype=D, generator=g)
    v = torch.randn(nkv, S, hd, dtype=D, generator=g)
    mask = torch.ones(T, S, dtype=torch.bool).tril(diagonal=S - T)
    ref = F.scaled_dot_product_attention(q[None], k.repeat_interleave(nq // nkv, 0)[None],
                                         v.repeat_interleave(nq // nkv, 0)[None], attn_mask=mask)[0]
    assert torch.allclose(of.causal_gqa_attention(q, k, v), ref, rtol=1e-12, atol=1e-13)


def test_attention_special_cases():
    g = torch.Generator().manual_seed(4)
    # one key: output is that key's value row, whatever the query
    q = torch.randn(4, 1, 8, dtype=D, generator=g)
    k = torch.randn(2, 1, 8, dtype=D, generator=g)
    v = torch.randn(2, 1, 8, dtype=D, generator=g)
    out = of.causal_gqa_attention(q, k, v)
    assert torch.allclose(out, v.repeat_interleave(2, 0), atol=1e-15)
    # zero query: uniform weights over the visible keys -> mean of visible values
    S, T = 9, 3
    k = torch.randn(1, S, 8, dtype=D, generator=g)
    v = torch.randn(1, S, 8, dtype=D, generator=g)
    out = of.causal_gqa_attention(torch.zeros(1, T, 8, dtype=D), k, v)
    for j in range(T):
        assert torch.allclose(out[0, j], v[0, : S - T + j + 1].mean(0), atol=1e-14)
    # causality: changing keys after the last visible one changes nothing
    q = torch.randn(2, T, 8, dtype=D, generator=g)
    k2, v2 = k.clone(), v.clone()
    k2[0, -1] += 5.0
    v2[0, -1] -= 3.0
    a = of.causal_gqa_attention(q, k.expand(2, -1, -1).contiguous()[:1], v[:1])
    b = of.causal_gqa_attention(q, k2[:1], v2[:1])
    assert torch.allclose(a[:, : T - 1], b[:, : T - 1], atol=0) and not torch.allclose(a[:, -1], b[:, -1])


def test_silu_and_argmax_semantics():
    z = torch.linspace(-20, 20, 101, dtype=D)
    assert torch.allclose(of.silu(z), F.silu(z), rtol=1e-14, atol=1e-300)
    x = torch.tensor([[1.0, 3.0, 3.0, 2.0], [0.0, float("nan"), 5.0, float("nan")], [-1.0, -1.0, -1.0, -1.0]], dtype=D)
    assert of.argmax_first(x).tolist() == torch.argmax(x, dim=-1).tolist() == [1, 1, 0]


def _tiny_weights(shape, seed):
    g = torch.Generator().manual_seed(seed)
    H, nq, nkv, hd, I = shape.hidden, shape.num_q_heads, shape.num_kv_heads, shape.head_dim, shape.intermediate
    r = lambda *s: torch.randn(*s, dtype=D, generator=g) * 0.3  # noqa: E731
    return of.LayerWeights(q=r(nq * hd, H), k=r(nkv * hd, H), v=r(nkv * hd, H), o=r(H, nq * hd),
                           gate=r(I, H), up=r(I, H), down=r(H, I),
                           in_norm=1 + r(H), post_norm=1 + r(H), q_norm=1 + r(hd), k_norm=1 + r(hd))


def _as_lists(w):
    return {k: getattr(w, k).tolist() for k in ("q", "k", "v", "o", "gate", "up", "down",
                                                "in_norm", "post_norm", "q_norm", "k_norm")}


TINY = of.Shape(hidden=32, num_q_heads=4, num_kv_heads=2, head_dim=8, intermediate=48, vocab=50,
                num_layers=1, rms_eps=1e-6, rope_theta=1e4)


def test_decoder_layer_matches_brute_force_loops():
    w = _tiny_weights(TINY, 5)
    g = torch.Generator().manual_seed(6)
    x = torch.randn(3, 32, dtype=D, generator=g)
    kc = torch.randn(2, 4, 8, dtype=D, generator=g)
    vc = torch.randn(2, 4, 8, dtype=D, generator=g)
    y, K, V = of.decoder_layer(x, w, TINY, kc, vc)
    by, bK, bV = brute.layer(x.tolist(), _as_lists(w), 4, 2, 8, TINY.rms_eps, TINY.rope_theta,
                             kc.tolist(), vc.tolist())
    assert torch.allclose(y, torch.tensor(by, dtype=D), rtol=1e-12, atol=1e-12)
    assert torch.allclose(K, torch.tensor(bK, dtype=D), atol=1e-13)
    assert torch.allclose(V, torch.tensor(bV, dtype=D), atol=0)


def test_cache_store_rounds_like_independent_bf16_conversions():
    """cache_store(x, bfloat16) is x rounded to fp32, then to bf16 with round to
    nearest, ties to even: checked against the input generator's bit-level rounding
    (numpy) and the brute-force scalar one, on random values and on exact ties
    (an odd last bf16 bit rounds up, an even one down)."""
    g = torch.Generator().manual_seed(11)
    x = torch.cat([torch.randn(10000, dtype=D, generator=g) * 3,
                   torch.tensor([1 + 2**-8, 1 + 3 * 2**-8, -(2 + 2**-7), 0.5 + 2**-10], dtype=D)])
    got = of.cache_store(x, torch.bfloat16)
    ref = synth.bf16_bits_to_f32(synth._f32_to_bf16_bits(x.numpy().astype(np.float32)))
    assert np.array_equal(got.numpy(), ref.astype(np.float64))
    assert [brute.bf16_value(float(v)) for v in x] == got.tolist()
    assert got[-4:].tolist() == [1.0, 1 + 4 * 2**-8, -2.0, 0.5]
    assert torch.equal(of.cache_store(x, None), x)


def test_bf16_cache_layer_matches_brute_force_loops():
    """With a bf16 cache the new K / V are stored rounded and attention reads the
    stored values: the layer equals the scalar loops that round what they append,
    the returned cache holds the rounded values, the trace the unrounded ones, and
    the output differs from that of a cache in full precision."""
    w = _tiny_weights(TINY, 5)
    g = torch.Generator().manual_seed(6)
    x = torch.randn(3, 32, dtype=D, generator=g)
    kc = of.cache_store(torch.randn(2, 4, 8, dtype=D, generator=g), torch.bfloat16)
    vc = of.cache_store(torch.randn(2, 4, 8, dtype=D, generator=g), torch.bfloat16)
    tr = {}
    y, K, V = of.decoder_layer(x, w, TINY, kc, vc, tr, torch.bfloat16)
    by, bK, bV = brute.layer(x.tolist(), _as_lists(w), 4, 2, 8, TINY.rms_eps, TINY.rope_theta,
                             kc.tolist(), vc.tolist(), store=brute.bf16_value)
    assert torch.allclose(y, torch.tensor(by, dtype=D), rtol=1e-12, atol=1e-12)
    assert torch.equal(K, torch.tensor(bK, dtype=D)) and torch.equal(V, torch.tensor(bV, dtype=D))
    assert torch.equal(K[:, 4:], of.cache_store(tr["k"], torch.bfloat16))
    assert torch.equal(V[:, 4:], of.cache_store(tr["v"], torch.bfloat16))
    assert not torch.equal(K[:, 4:], tr["k"])
    y_full, _, _ = of.decoder_layer(x, w, TINY, kc, vc)
    assert float((y - y_full).abs().max()) > 1e-6


def test_head_matches_brute_force():
    g = torch.Generator().manual_seed(7)
    hw = of.HeadWeights(embed=torch.randn(50, 32, dtype=D, generator=g), lm_head=None,
                        final_norm=1 + 0.1 * torch.randn(32, dtype=D, generator=g))
    hw.lm_head = hw.embed
    x = torch.randn(32, dtype=D, generator=g)
    logits = of.lm_head(x, hw, TINY)
    bl, bi = brute.head_argmax(x.tolist(), hw.final_norm.tolist(), hw.lm_head.tolist(), TINY.rms_eps)
    assert torch.allclose(logits, torch.tensor(bl, dtype=D), rtol=1e-13, atol=1e-13)
    assert int(of.argmax_first(logits)) == bi
    ids = torch.tensor([0, 49, 7, 7])
    assert torch.equal(of.embed(ids, hw), hw.embed[[0, 49, 7, 7]])


@pytest.mark.slow
def test_tiny_workload_layer_matches_brute_force():
    """The tiny workload (hidden 256, 4 q / 2 kv heads, hd 64) with generated
    bf16 weights and perturbed norms, one layer over 8 prefill tokens."""
    s = synth.TINY
    shape = oi.shape_of(s)
    w = oi.layer_weights(s, 0, perturbed_norms=True)
    x = of.from_bf16_bits(synth.hidden_bits(8, s.hidden))
    empty = torch.zeros(2, 0, 64, dtype=D)
    y, _, _ = of.decoder_layer(x, w, shape, empty, empty)
    by, _, _ = brute.layer(x.tolist(), _as_lists(w), 4, 2, 64, s.rms_eps, s.rope_theta, [[], []], [[], []])
    assert torch.allclose(y, torch.tensor(by, dtype=D), rtol=1e-11, atol=1e-12)
