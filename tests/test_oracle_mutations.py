"""Planted mistakes in the oracle (CPU only): each plausible slip must make one
of the pins fail, so that the pins are known to have teeth."""

import math

import pytest
import torch

from oracle import brute
from oracle import forward as of
from tests.test_oracle_pins import TINY, _as_lists, _tiny_weights

D = torch.float64


def _layer_vs_brute():
    w = _tiny_weights(TINY, 31)
    g = torch.Generator().manual_seed(32)
    x = torch.randn(3, 32, dtype=D, generator=g)
    kc = torch.randn(2, 2, 8, dtype=D, generator=g)
    vc = torch.randn(2, 2, 8, dtype=D, generator=g)
    y, _, _ = of.decoder_layer(x, w, TINY, kc, vc)
    by, _, _ = brute.layer(x.tolist(), _as_lists(w), 4, 2, 8, TINY.rms_eps, TINY.rope_theta,
                           kc.tolist(), vc.tolist())
    return torch.allclose(y, torch.tensor(by, dtype=D), rtol=1e-10, atol=1e-10)


def test_unmodified_oracle_agrees():
    assert _layer_vs_brute()


def _wrong_rope_sign(u, positions, theta):
    hd = u.shape[-1]
    ang = of.rope_angles(positions, hd, theta, torch.float64)
    cos, sin = torch.cos(ang), torch.sin(ang)
    a, b = u[..., : hd // 2], u[..., hd // 2:]
    return torch.cat([a * cos + b * sin, b * cos - a * sin], dim=-1)


def _rms_no_eps(x, w, eps):
    return x / torch.sqrt((x * x).mean(-1, keepdim=True)) * w


def _rms_no_weight(x, w, eps):
    return x / torch.sqrt((x * x).mean(-1, keepdim=True) + eps)


def _attn_no_scale(q, k, v):
    return of_causal(q * math.sqrt(q.shape[-1]), k, v)


def _attn_wrong_gqa(q, k, v):
    # repeat instead of repeat_interleave: head h reads kv head h % nkv
    nq, nkv = q.shape[0], k.shape[0]
    return of_causal(q, k.repeat(nq // nkv, 1, 1), v.repeat(nq // nkv, 1, 1))


def _attn_no_offset(q, k, v):
    T, S = q.shape[1], k.shape[1]
    kk = k.repeat_interleave(q.shape[0] // k.shape[0], 0)
    vv = v.repeat_interleave(q.shape[0] // k.shape[0], 0)
    s = (q @ kk.transpose(-1, -2)) / math.sqrt(q.shape[-1])
    s = s.masked_fill(~torch.ones(T, S, dtype=torch.bool).tril(), float("-inf"))
    return torch.softmax(s, -1) @ vv


def _silu_as_sigmoid(z):
    return 1.0 / (1.0 + torch.exp(-z))


of_causal = of.causal_gqa_attention


@pytest.mark.parametrize("name,patch", [
    ("apply_rope", _wrong_rope_sign),
    ("rms_norm", _rms_no_eps),
    ("rms_norm", _rms_no_weight),
    ("causal_gqa_attention", _attn_no_scale),
    ("causal_gqa_attention", _attn_wrong_gqa),
    ("causal_gqa_attention", _attn_no_offset),
    ("silu", _silu_as_sigmoid),
])
def test_planted_mistake_is_caught(monkeypatch, name, patch):
    monkeypatch.setattr(of, name, patch)
    assert not _layer_vs_brute()


def test_planted_shard_slip_is_caught():
    """A rank taking the wrong kv head (r * nkv // n off by one) breaks sharded == unsharded."""
    shape = of.Shape(hidden=32, num_q_heads=8, num_kv_heads=2, head_dim=4, intermediate=32, vocab=40,
                     num_layers=1)
    g = torch.Generator().manual_seed(33)
    r = lambda *s: torch.randn(*s, dtype=D, generator=g) * 0.3  # noqa: E731
    w = of.LayerWeights(q=r(32, 32), k=r(8, 32), v=r(8, 32), o=r(32, 32), gate=r(32, 32), up=r(32, 32),
                        down=r(32, 32), in_norm=1 + r(32), post_norm=1 + r(32), q_norm=1 + r(4), k_norm=1 + r(4))
    x = torch.randn(3, 32, dtype=D, generator=g)
    empty = torch.zeros(2, 0, 4, dtype=D)
    ref, _, _ = of.decoder_layer(x, w, shape, empty, empty)

    def run():
        ranks = [of.shard_layer(w, shape, 4, rr) for rr in range(4)]
        caches = of.split_kv_by_rank(empty, shape, 4)
        y, _, _ = of.tp_decoder_layer(x, ranks, shape, caches, caches, of.Comm())
        return torch.allclose(y, ref, atol=1e-12)

    assert run()
    orig = of.kv_heads_of_rank
    try:
        of.kv_heads_of_rank = lambda s, n, rr: [min(s.num_kv_heads - 1, (rr + 1) * s.num_kv_heads // n)]
        assert not run()
    finally:
        of.kv_heads_of_rank = orig
