"""Glue from the seeded generator (``synth``) to oracle tensors.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  Converts the shared
generator's bf16 bit patterns into float tensors; no arithmetic of the method.
"""

from __future__ import annotations

from typing import List, Optional, Sequence

import numpy as np
import torch

import synth
from oracle.forward import DTYPE, HeadWeights, LayerWeights, SeqInput, Shape, from_bf16_bits


def shape_of(s: synth.ModelShape, num_layers: Optional[int] = None) -> Shape:
    return Shape(hidden=s.hidden, num_q_heads=s.num_q_heads, num_kv_heads=s.num_kv_heads,
                 head_dim=s.head_dim, intermediate=s.intermediate, vocab=s.vocab,
                 num_layers=s.num_layers if num_layers is None else num_layers,
                 rms_eps=s.rms_eps, rope_theta=s.rope_theta,
                 tie_word_embeddings=s.tie_word_embeddings)


def layer_weights(s: synth.ModelShape, layer: int, perturbed_norms: bool = False,
                  dtype=DTYPE) -> LayerWeights:
    g = lambda kind: from_bf16_bits(synth.layer_weight_bits(s, layer, kind, perturbed_norms), dtype)  # noqa: E731
    return LayerWeights(q=g(synth.W_Q), k=g(synth.W_K), v=g(synth.W_V), o=g(synth.W_O),
                        gate=g(synth.W_GATE), up=g(synth.W_UP), down=g(synth.W_DOWN),
                        in_norm=g(synth.W_IN_NORM), post_norm=g(synth.W_POST_NORM),
                        q_norm=g(synth.W_Q_NORM), k_norm=g(synth.W_K_NORM))


def head_weights(s: synth.ModelShape, perturbed_norms: bool = False, dtype=DTYPE,
                 need_embed: bool = True) -> HeadWeights:
    """The embedding, LM head and final norm.  need_embed=False leaves out an
    untied embedding table (for steps that start from hidden states)."""
    tied = s.tie_word_embeddings
    emb = from_bf16_bits(synth.global_weight_bits(s, synth.W_EMBED), dtype) if (tied or need_embed) else None
    lm = emb if tied else from_bf16_bits(synth.global_weight_bits(s, synth.W_LM_HEAD), dtype)
    fn = from_bf16_bits(synth.global_weight_bits(s, synth.W_FINAL_NORM, perturbed_norms), dtype)
    return HeadWeights(embed=emb, lm_head=lm, final_norm=fn)


def cached_kv(s: synth.ModelShape, layer: int, slot: int, ctx: int, dtype=DTYPE):
    """Synthetic cached K and V [nkv, ctx, hd] of one sequence slot for one layer."""
    ks = [from_bf16_bits(synth.kv_cache_bits(layer, slot, 0, g, ctx, s.num_kv_heads, s.head_dim), dtype)
          for g in range(s.num_kv_heads)]
    vs = [from_bf16_bits(synth.kv_cache_bits(layer, slot, 1, g, ctx, s.num_kv_heads, s.head_dim), dtype)
          for g in range(s.num_kv_heads)]
    if ctx == 0:
        empty = torch.zeros(s.num_kv_heads, 0, s.head_dim, dtype=dtype)
        return empty, empty.clone()
    return torch.stack(ks), torch.stack(vs)


def workload_seq_inputs(w: synth.Workload, seqs: Sequence[int], layers: Sequence[int],
                        dtype=DTYPE) -> List[SeqInput]:
    """Inputs of the chosen sequences of a workload step (sequence b uses cache slot b)."""
    s = w.shape
    q_lens, ctx_lens = w.q_lens, w.ctx_lens
    cu = np.concatenate([[0], np.cumsum(q_lens)])
    out = []
    ids_all = synth.step_token_ids(w.num_tokens, s.vocab) if w.input_from_ids else None
    for b in seqs:
        t0, t1 = int(cu[b]), int(cu[b + 1])
        hidden = ids = None
        if w.input_from_ids:
            ids = torch.from_numpy(ids_all[t0:t1].copy())
        else:
            hidden = from_bf16_bits(synth.normal_bf16_bits(synth.SEED_ACTIVATIONS, 0, (t1 - t0) * s.hidden,
                                                           1.0, start=t0 * s.hidden), dtype).reshape(t1 - t0, s.hidden)
        kc, vc = [], []
        for li in layers:
            k, v = cached_kv(s, li, b, ctx_lens[b], dtype)
            kc.append(k)
            vc.append(v)
        out.append(SeqInput(hidden=hidden, ids=ids, k_cache=kc, v_cache=vc))
    return out
