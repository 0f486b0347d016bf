"""Unsharded reference forward and the tensor-parallel emulation (CPU, plain torch).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  Everything computes in
``dtype`` (float64 unless a test asks for float32), from bf16 weight bits
upcast exactly.  No blocking, fusion or reordering beyond what each definition
states; library calls are limited to matmul and elementwise math.

Readings taken where the pages are silent:
  * RMSNorm is x / sqrt(mean(x^2) + eps) * w (the pages import it, never show it).
  * RoPE is the rotate-half form: for d < hd/2, angle = p * theta^(-2d/hd),
    (a, b) = (u[d], u[d + hd/2]) -> (a cos - b sin, b cos + a sin).
  * q/k RMSNorm per head over head_dim comes before RoPE; the cache keeps
    post-RoPE K and raw V.
  * Attention scale 1/sqrt(hd); query j of a step with T new tokens over S
    keys may see keys 0 .. j + (S - T).
  * Uneven splits are errors (no silent short chunks); vocab slices use
    div_ceil and the last slice may be shorter, but none may be empty.
  * The KV cache holds values in its own element type (``kv_dtype``): None keeps
    the computing precision (the pages' fp32 demo), torch.bfloat16 is the bf16
    cache the workloads name.  New K/V are rounded when appended (via fp32, round
    to nearest even at each step) and attention reads what the cache holds, as
    it does in tp.py (the cache is updated, then attention reads the cache).
  * Sequence parallelism splits the tokens into contiguous rank chunks as even
    as possible, the first T mod n ranks taking one token more (a rank may get
    none); the final norm runs on the chunks and an all-gather of the normed
    rows feeds the vocab-parallel head, as before any column-split layer.
  * No bias anywhere.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np
import torch

DTYPE = torch.float64


# ---------------------------------------------------------------------------
# bf16 bits -> float
# ---------------------------------------------------------------------------

def from_bf16_bits(bits: np.ndarray, dtype=DTYPE) -> torch.Tensor:
    """Exact upcast of bf16 bit patterns (uint16) to ``dtype``."""
    u32 = np.left_shift(np.asarray(bits, dtype=np.uint16).astype(np.uint32), np.uint32(16))
    return torch.from_numpy(u32.view(np.float32).copy()).to(dtype)


# ---------------------------------------------------------------------------
# Model shape and weights
# ---------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class Shape:
    hidden: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    intermediate: int
    vocab: int
    num_layers: int
    rms_eps: float = 1e-6
    rope_theta: float = 1e6
    tie_word_embeddings: bool = True


@dataclasses.dataclass
class LayerWeights:
    """Full (unsharded) tensors of one decoder layer, nn.Linear layout [out, in]."""
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    o: torch.Tensor
    gate: torch.Tensor
    up: torch.Tensor
    down: torch.Tensor
    in_norm: torch.Tensor
    post_norm: torch.Tensor
    q_norm: torch.Tensor
    k_norm: torch.Tensor


@dataclasses.dataclass
class HeadWeights:
    embed: torch.Tensor        # [V, H]
    lm_head: torch.Tensor      # [V, H]; the same tensor as ``embed`` when tied
    final_norm: torch.Tensor   # [H]


# ---------------------------------------------------------------------------
# Building blocks ([TP] "Implementation": tp.py imports RMSNorm, apply_rope,
# rope_cos_sin from mini_llm without showing them; readings in the header)
# ---------------------------------------------------------------------------

def rms_norm(x: torch.Tensor, w: torch.Tensor, eps: float) -> torch.Tensor:
    """RMSNorm over the last dimension: x / sqrt(mean(x^2) + eps) * w."""
    ms = (x * x).mean(dim=-1, keepdim=True)
    return x / torch.sqrt(ms + eps) * w


def rope_angles(positions: torch.Tensor, head_dim: int, theta: float, dtype=DTYPE) -> torch.Tensor:
    """angle[p, d] = p * theta^(-2d/head_dim) for d < head_dim/2 (rotary frequencies)."""
    d = torch.arange(head_dim // 2, dtype=torch.float64)
    inv_freq = theta ** (-2.0 * d / head_dim)
    return (positions.to(torch.float64)[:, None] * inv_freq[None, :]).to(dtype)


def apply_rope(u: torch.Tensor, positions: torch.Tensor, theta: float) -> torch.Tensor:
    """Rotate-half RoPE on the last dim of u [..., T, hd] at the given positions [T].

    The pair (u[d], u[d + hd/2]) is rotated by angle(p, d):
    (a, b) -> (a cos - b sin, b cos + a sin).   ([TP] TPAttention.forward: q and k
    get RoPE at positions start .. start + T, after q_norm/k_norm.)
    """
    hd = u.shape[-1]
    ang = rope_angles(positions, hd, theta, torch.float64)
    cos, sin = torch.cos(ang).to(u.dtype), torch.sin(ang).to(u.dtype)
    a, b = u[..., : hd // 2], u[..., hd // 2:]
    return torch.cat([a * cos - b * sin, b * cos + a * sin], dim=-1)


def cache_store(x: torch.Tensor, kv_dtype: Optional[torch.dtype]) -> torch.Tensor:
    """The values a KV cache of element type ``kv_dtype`` holds for ``x``: x itself
    when kv_dtype is None, else x rounded to fp32 and then to kv_dtype (round to
    nearest, ties to even) and read back exactly."""
    if kv_dtype is None:
        return x
    return x.to(torch.float32).to(kv_dtype).to(x.dtype)


def silu(z: torch.Tensor) -> torch.Tensor:
    """silu(z) = z * sigmoid(z) = z / (1 + exp(-z))."""
    return z / (1.0 + torch.exp(-z))


def causal_gqa_attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor) -> torch.Tensor:
    """softmax(q k^T / sqrt(hd) + mask) v with GQA and a cache offset.

    q [nq, T, hd] (the T newest positions), k/v [nkv, S, hd] (all S positions,
    cache first).  Query head h reads kv head h // (nq / nkv) (repeat_interleave).
    Query j may see keys 0 .. j + (S - T) (tril with diagonal S - T).
    ([TP] TPAttention.forward.)
    """
    nq, T, hd = q.shape
    nkv, S, _ = k.shape
    rep = nq // nkv
    k = k.repeat_interleave(rep, dim=0)
    v = v.repeat_interleave(rep, dim=0)
    scores = (q @ k.transpose(-1, -2)) / math.sqrt(hd)
    allowed = torch.ones(T, S, dtype=torch.bool).tril(diagonal=S - T)
    scores = scores.masked_fill(~allowed, float("-inf"))
    m = scores.max(dim=-1, keepdim=True).values
    e = torch.exp(scores - m)
    p = e / e.sum(dim=-1, keepdim=True)
    return p @ v


def argmax_first(logits: torch.Tensor) -> torch.Tensor:
    """Index of the maximum along the last dim; the first one on ties; NaN counts
    as the maximum (torch.argmax semantics, [TP] main: logits[0, -1].argmax())."""
    x = logits
    nan = torch.isnan(x)
    out = []
    for row, nrow in zip(x.reshape(-1, x.shape[-1]), nan.reshape(-1, x.shape[-1])):
        if bool(nrow.any()):
            out.append(int(torch.nonzero(nrow)[0]))
            continue
        mx = row.max()
        out.append(int(torch.nonzero(row == mx)[0]))
    return torch.tensor(out, dtype=torch.int64).reshape(x.shape[:-1])


# ---------------------------------------------------------------------------
# Unsharded forward (one sequence at a time)
# ---------------------------------------------------------------------------

def decoder_layer(x: torch.Tensor, w: LayerWeights, shape: Shape,
                  k_cache: torch.Tensor, v_cache: torch.Tensor, trace: Optional[dict] = None,
                  kv_dtype: Optional[torch.dtype] = None) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """One decoder layer for one sequence, unsharded.

    x [T, H] are the sequence's T new tokens at positions ctx .. ctx+T-1 where
    ctx = k_cache.shape[1]; k_cache/v_cache [nkv, ctx, hd].  Returns the new
    hidden [T, H] and the caches extended by T positions (the new K and V as a
    cache of element type kv_dtype holds them; ``trace`` gets them unrounded).
    ([TP] TPTransformer.forward loop body: x = x + attn(ln1(x)); x = x + mlp(ln2(x)).)
    """
    T = x.shape[0]
    nq, nkv, hd = shape.num_q_heads, shape.num_kv_heads, shape.head_dim
    ctx = k_cache.shape[1]
    pos = torch.arange(ctx, ctx + T)
    h = rms_norm(x, w.in_norm, shape.rms_eps)
    q = (h @ w.q.T).reshape(T, nq, hd).transpose(0, 1)
    k = (h @ w.k.T).reshape(T, nkv, hd).transpose(0, 1)
    v = (h @ w.v.T).reshape(T, nkv, hd).transpose(0, 1)
    q = rms_norm(q, w.q_norm, shape.rms_eps)
    k = rms_norm(k, w.k_norm, shape.rms_eps)
    q = apply_rope(q, pos, shape.rope_theta)
    k = apply_rope(k, pos, shape.rope_theta)
    K = torch.cat([k_cache, cache_store(k, kv_dtype)], dim=1)
    V = torch.cat([v_cache, cache_store(v, kv_dtype)], dim=1)
    o = causal_gqa_attention(q, K, V)
    x = x + o.transpose(0, 1).reshape(T, nq * hd) @ w.o.T
    h2 = rms_norm(x, w.post_norm, shape.rms_eps)
    act = silu(h2 @ w.gate.T) * (h2 @ w.up.T)
    if trace is not None:  # intermediates, for diagnosis only
        trace.update(h=h, q=q, k=k, v=v, attn=o.transpose(0, 1).reshape(T, nq * hd), x_mid=x, h2=h2, act=act)
    x = x + act @ w.down.T
    return x, K, V


def embed(ids: torch.Tensor, hw: HeadWeights) -> torch.Tensor:
    """x_t = E[id_t] (plain row lookup)."""
    return hw.embed[ids]


def lm_head(x_last: torch.Tensor, hw: HeadWeights, shape: Shape) -> torch.Tensor:
    """logits = RMSNorm(x_last; w_final) LM^T for the last position of each sequence
    ([TP] TPTransformer.forward: norm(x[:, -1:]) then the output layer)."""
    return rms_norm(x_last, hw.final_norm, shape.rms_eps) @ hw.lm_head.T


# ---------------------------------------------------------------------------
# Shard rules ([SHD] weight.py:13-14, 34-52; [TP] "KV heads and the limit on TP")
# ---------------------------------------------------------------------------

class ShardError(ValueError):
    pass


def div_ceil(a: int, b: int) -> int:
    return (a + b - 1) // b


def validate_tp(shape: Shape, n: int) -> None:
    """Reject tp sizes the pages rule out, and uneven splits (read as errors)."""
    if n < 1:
        raise ShardError("tp_size must be >= 1")
    if shape.num_q_heads % n:
        raise ShardError(f"{shape.num_q_heads} query heads are not divisible by tp_size {n}")
    nkv = shape.num_kv_heads
    if nkv >= n and nkv % n:
        raise ShardError(f"{nkv} kv heads are not divisible by tp_size {n}")
    if nkv < n and n % nkv:
        raise ShardError(f"tp_size {n} is not a multiple of {nkv} kv heads (replication)")
    if shape.intermediate % n:
        raise ShardError(f"intermediate {shape.intermediate} is not divisible by tp_size {n}")
    per = div_ceil(shape.vocab, n)
    if (n - 1) * per >= shape.vocab:
        raise ShardError(f"vocab {shape.vocab} leaves rank {n - 1} an empty slice at tp_size {n}")


def vocab_range(vocab: int, n: int, r: int) -> Tuple[int, int]:
    """[start, end) of rank r's vocabulary slice: per = div_ceil(V, n)."""
    per = div_ceil(vocab, n)
    return r * per, min((r + 1) * per, vocab)


def even_chunk(size: int, n: int, r: int) -> Tuple[int, int]:
    """torch.chunk(n)[r] on a dimension divisible by n."""
    if size % n:
        raise ShardError(f"dimension {size} is not divisible by {n}")
    c = size // n
    return r * c, (r + 1) * c


def token_chunk(T: int, n: int, r: int) -> Tuple[int, int]:
    """[start, end) of rank r's tokens under sequence parallelism: contiguous,
    as even as possible, the first T mod n ranks one token more."""
    base, extra = divmod(T, n)
    start = r * base + min(r, extra)
    return start, start + base + (1 if r < extra else 0)


def kv_heads_of_rank(shape: Shape, n: int, r: int) -> List[int]:
    """Global kv heads held by rank r: an even chunk, or, when there are fewer kv
    heads than ranks, the single head r * nkv // n (replicated on several ranks)."""
    nkv = shape.num_kv_heads
    if nkv < n:
        return [r * nkv // n]
    a, b = even_chunk(nkv, n, r)
    return list(range(a, b))


SPLIT_ROWS = ("q", "k", "v", "gate", "up")    # _SPLIT_DIM_0
SPLIT_COLS = ("o", "down")                     # _SPLIT_DIM_1


def shard_index(kind: str, shape: Shape, n: int, r: int) -> Tuple[str, np.ndarray]:
    """Which dimension of the full tensor rank r takes, and the source indices.

    Returns ("rows" | "cols" | "all", int64 indices).  q/k/v/gate/up take rows,
    o/down take columns, embed/lm_head take a div_ceil vocab slice of rows,
    norms are kept whole.
    """
    hd = shape.head_dim
    if kind in ("k", "v"):
        heads = kv_heads_of_rank(shape, n, r)
        rows = np.concatenate([np.arange(g * hd, (g + 1) * hd) for g in heads])
        return "rows", rows.astype(np.int64)
    if kind == "q":
        a, b = even_chunk(shape.num_q_heads * hd, n, r)
        return "rows", np.arange(a, b, dtype=np.int64)
    if kind in ("gate", "up"):
        a, b = even_chunk(shape.intermediate, n, r)
        return "rows", np.arange(a, b, dtype=np.int64)
    if kind == "o":
        a, b = even_chunk(shape.num_q_heads * hd, n, r)
        return "cols", np.arange(a, b, dtype=np.int64)
    if kind == "down":
        a, b = even_chunk(shape.intermediate, n, r)
        return "cols", np.arange(a, b, dtype=np.int64)
    if kind in ("embed", "lm_head"):
        a, b = vocab_range(shape.vocab, n, r)
        return "rows", np.arange(a, b, dtype=np.int64)
    if kind in ("in_norm", "post_norm", "q_norm", "k_norm", "final_norm"):
        size = shape.head_dim if kind in ("q_norm", "k_norm") else shape.hidden
        return "all", np.arange(size, dtype=np.int64)
    raise KeyError(kind)


def shard_tensor(kind: str, full: torch.Tensor, shape: Shape, n: int, r: int) -> torch.Tensor:
    dim, idx = shard_index(kind, shape, n, r)
    t = torch.from_numpy(idx)
    if dim == "rows":
        return full[t].clone()
    if dim == "cols":
        return full[:, t].clone()
    return full.clone()


@dataclasses.dataclass
class RankLayer:
    """Rank r's weights of one layer after shard-then-merge ([CH9] 3.3)."""
    qkv: torch.Tensor       # cat(q_r, k_r, v_r) along rows
    gate_up: torch.Tensor   # cat(gate_r, up_r) along rows
    o: torch.Tensor         # [H, nq_l * hd]
    down: torch.Tensor      # [H, I_l]
    in_norm: torch.Tensor
    post_norm: torch.Tensor
    q_norm: torch.Tensor
    k_norm: torch.Tensor
    nq_l: int
    nkv_l: int
    i_l: int
    kv_heads: List[int]


def shard_layer(w: LayerWeights, shape: Shape, n: int, r: int) -> RankLayer:
    validate_tp(shape, n)
    sh = lambda kind, t: shard_tensor(kind, t, shape, n, r)  # noqa: E731
    q, k, v = sh("q", w.q), sh("k", w.k), sh("v", w.v)
    g, u = sh("gate", w.gate), sh("up", w.up)
    heads = kv_heads_of_rank(shape, n, r)
    return RankLayer(qkv=torch.cat([q, k, v], dim=0), gate_up=torch.cat([g, u], dim=0),
                     o=sh("o", w.o), down=sh("down", w.down),
                     in_norm=sh("in_norm", w.in_norm), post_norm=sh("post_norm", w.post_norm),
                     q_norm=sh("q_norm", w.q_norm), k_norm=sh("k_norm", w.k_norm),
                     nq_l=shape.num_q_heads // n, nkv_l=len(heads), i_l=g.shape[0], kv_heads=heads)


# ---------------------------------------------------------------------------
# Tensor-parallel emulation: every rank computes locally, the only cross-rank
# steps are the counted sums (all-reduce) and the logits gather (all-gather).
# ---------------------------------------------------------------------------

class Comm:
    """Stands in for the collectives: a rank-ordered sum and a gather, counted;
    for sequence parallelism also the sum scattered by token chunk and the
    gather of token chunks."""

    def __init__(self) -> None:
        self.num_all_reduce = 0
        self.num_all_gather = 0
        self.num_reduce_scatter = 0
        self.num_all_gather_rows = 0

    def reduce_scatter(self, partials: Sequence[torch.Tensor]) -> List[torch.Tensor]:
        """Rank r receives the rank-ordered sum of rows token_chunk(T, n, r)."""
        self.num_reduce_scatter += 1
        n, T = len(partials), partials[0].shape[0]
        out = []
        for r in range(n):
            a, b = token_chunk(T, n, r)
            acc = partials[0][a:b].clone()
            for p in partials[1:]:
                acc = acc + p[a:b]
            out.append(acc)
        return out

    def all_gather_rows(self, chunks: Sequence[torch.Tensor]) -> torch.Tensor:
        """Every rank receives the token chunks of all ranks, in rank order."""
        self.num_all_gather_rows += 1
        return torch.cat(list(chunks), dim=0)

    def all_reduce(self, partials: Sequence[torch.Tensor]) -> torch.Tensor:
        self.num_all_reduce += 1
        acc = partials[0].clone()
        for p in partials[1:]:
            acc = acc + p
        return acc

    def all_gather(self, parts: Sequence[torch.Tensor]) -> torch.Tensor:
        self.num_all_gather += 1
        return torch.cat(list(parts), dim=-1)


def tp_embed(ids: torch.Tensor, hw: HeadWeights, shape: Shape, n: int, comm: Comm) -> torch.Tensor:
    """Vocab-parallel embedding: each rank looks up ids in its slice, ids outside
    the slice give 0, then the partials are summed ([TP] VocabParallelEmbedding)."""
    partials = []
    for r in range(n):
        start, end = vocab_range(shape.vocab, n, r)
        e_r = shard_tensor("embed", hw.embed, shape, n, r)
        outside = (ids < start) | (ids >= end)
        local = (ids - start).masked_fill(outside, 0)
        y = e_r[local].masked_fill(outside[..., None], 0.0)
        partials.append(y)
    return comm.all_reduce(partials)


def tp_decoder_layer(x: torch.Tensor, ranks: Sequence[RankLayer], shape: Shape,
                     k_caches: Sequence[torch.Tensor], v_caches: Sequence[torch.Tensor], comm: Comm,
                     kv_dtype: Optional[torch.dtype] = None
                     ) -> Tuple[torch.Tensor, List[torch.Tensor], List[torch.Tensor]]:
    """One layer under tensor parallelism for one sequence.

    Column-split q/k/v and gate/up need no exchange; the row-split o_proj and
    down_proj each give per-rank partials that one all-reduce sums
    ([TP] TPAttention / TPMLP; [SHD] linear.py:102-106).  k_caches[r] and
    v_caches[r] [nkv_l, ctx, hd] hold rank r's kv heads.
    """
    T = x.shape[0]
    hd, eps = shape.head_dim, shape.rms_eps
    attn_partials, new_k, new_v = [], [], []
    for r, rl in enumerate(ranks):
        ctx = k_caches[r].shape[1]
        pos = torch.arange(ctx, ctx + T)
        h = rms_norm(x, rl.in_norm, eps)
        qkv = h @ rl.qkv.T
        nq_w, nkv_w = rl.nq_l * hd, rl.nkv_l * hd
        q = qkv[:, :nq_w].reshape(T, rl.nq_l, hd).transpose(0, 1)
        k = qkv[:, nq_w:nq_w + nkv_w].reshape(T, rl.nkv_l, hd).transpose(0, 1)
        v = qkv[:, nq_w + nkv_w:].reshape(T, rl.nkv_l, hd).transpose(0, 1)
        q = apply_rope(rms_norm(q, rl.q_norm, eps), pos, shape.rope_theta)
        k = apply_rope(rms_norm(k, rl.k_norm, eps), pos, shape.rope_theta)
        K = torch.cat([k_caches[r], cache_store(k, kv_dtype)], dim=1)
        V = torch.cat([v_caches[r], cache_store(v, kv_dtype)], dim=1)
        o = causal_gqa_attention(q, K, V)
        attn_partials.append(o.transpose(0, 1).reshape(T, nq_w) @ rl.o.T)
        new_k.append(K)
        new_v.append(V)
    x = x + comm.all_reduce(attn_partials)
    mlp_partials = []
    for rl in ranks:
        h2 = rms_norm(x, rl.post_norm, eps)
        gu = h2 @ rl.gate_up.T
        a = silu(gu[:, : rl.i_l]) * gu[:, rl.i_l:]
        mlp_partials.append(a @ rl.down.T)
    x = x + comm.all_reduce(mlp_partials)
    return x, new_k, new_v


def tp_lm_head(x_last: torch.Tensor, hw: HeadWeights, shape: Shape, n: int, comm: Comm) -> torch.Tensor:
    """Vocab-parallel logits: each rank computes its slice (padded to div_ceil(V, n)
    columns), an all-gather joins them and the result is truncated to V
    ([TP] TPTransformer.forward; [CH9] ParallelLMHead)."""
    per = div_ceil(shape.vocab, n)
    z = rms_norm(x_last, hw.final_norm, shape.rms_eps)
    parts = []
    for r in range(n):
        lm_r = shard_tensor("lm_head", hw.lm_head, shape, n, r)
        local = z @ lm_r.T
        if local.shape[-1] < per:
            pad = torch.zeros(*local.shape[:-1], per - local.shape[-1], dtype=local.dtype)
            local = torch.cat([local, pad], dim=-1)
        parts.append(local)
    return comm.all_gather(parts)[..., : shape.vocab]


# ---------------------------------------------------------------------------
# Sequence parallelism ("Tensor parallelism from scratch", section "Exercises",
# exercise 1): each all-reduce after a row-split GEMM becomes a reduce-scatter
# to the ranks' token chunks; the residual add and the RMSNorm run on a rank's
# own tokens only; an all-gather of the normed chunks precedes each
# column-split GEMM.  The collectives move the same data as the all-reduce
# they replace; the per-token work of each rank drops to its 1/n of the tokens.
# ---------------------------------------------------------------------------

def sp_embed(ids: torch.Tensor, hw: HeadWeights, shape: Shape, n: int, comm: Comm) -> List[torch.Tensor]:
    """Vocab-parallel embedding whose rank sum is scattered by token chunk."""
    partials = []
    for r in range(n):
        start, end = vocab_range(shape.vocab, n, r)
        e_r = shard_tensor("embed", hw.embed, shape, n, r)
        outside = (ids < start) | (ids >= end)
        local = (ids - start).masked_fill(outside, 0)
        partials.append(e_r[local].masked_fill(outside[..., None], 0.0))
    return comm.reduce_scatter(partials)


def sp_decoder_layer(x_chunks: Sequence[torch.Tensor], ranks: Sequence[RankLayer], shape: Shape,
                     k_caches: Sequence[torch.Tensor], v_caches: Sequence[torch.Tensor], comm: Comm,
                     kv_dtype: Optional[torch.dtype] = None
                     ) -> Tuple[List[torch.Tensor], List[torch.Tensor], List[torch.Tensor]]:
    """One layer under tensor + sequence parallelism for one sequence.  Rank r
    holds x_chunks[r], the residual rows of its token chunk; the column GEMMs
    and attention see all tokens (gathered), the row GEMMs' partials are
    summed into the chunks."""
    eps, hd = shape.rms_eps, shape.head_dim
    h = comm.all_gather_rows([rms_norm(x_chunks[r], ranks[r].in_norm, eps) for r in range(len(ranks))])
    T = h.shape[0]
    attn_partials, new_k, new_v = [], [], []
    for r, rl in enumerate(ranks):
        ctx = k_caches[r].shape[1]
        pos = torch.arange(ctx, ctx + T)
        qkv = h @ rl.qkv.T
        nq_w, nkv_w = rl.nq_l * hd, rl.nkv_l * hd
        q = qkv[:, :nq_w].reshape(T, rl.nq_l, hd).transpose(0, 1)
        k = qkv[:, nq_w:nq_w + nkv_w].reshape(T, rl.nkv_l, hd).transpose(0, 1)
        v = qkv[:, nq_w + nkv_w:].reshape(T, rl.nkv_l, hd).transpose(0, 1)
        q = apply_rope(rms_norm(q, rl.q_norm, eps), pos, shape.rope_theta)
        k = apply_rope(rms_norm(k, rl.k_norm, eps), pos, shape.rope_theta)
        K = torch.cat([k_caches[r], cache_store(k, kv_dtype)], dim=1)
        V = torch.cat([v_caches[r], cache_store(v, kv_dtype)], dim=1)
        o = causal_gqa_attention(q, K, V)
        attn_partials.append(o.transpose(0, 1).reshape(T, nq_w) @ rl.o.T)
        new_k.append(K)
        new_v.append(V)
    x_chunks = [x + s for x, s in zip(x_chunks, comm.reduce_scatter(attn_partials))]
    h2 = comm.all_gather_rows([rms_norm(x_chunks[r], ranks[r].post_norm, eps) for r in range(len(ranks))])
    mlp_partials = []
    for rl in ranks:
        gu = h2 @ rl.gate_up.T
        a = silu(gu[:, : rl.i_l]) * gu[:, rl.i_l:]
        mlp_partials.append(a @ rl.down.T)
    x_chunks = [x + s for x, s in zip(x_chunks, comm.reduce_scatter(mlp_partials))]
    return x_chunks, new_k, new_v


def sp_lm_head(x_chunks: Sequence[torch.Tensor], hw: HeadWeights, shape: Shape, n: int, comm: Comm) -> torch.Tensor:
    """Final norm on each rank's chunk, all-gather of the normed rows, then the
    vocab-parallel logits of the last position (tp_lm_head's slices and gather)."""
    z = comm.all_gather_rows([rms_norm(x, hw.final_norm, shape.rms_eps) for x in x_chunks])[-1]
    parts = []
    per = div_ceil(shape.vocab, n)
    for r in range(n):
        local = z @ shard_tensor("lm_head", hw.lm_head, shape, n, r).T
        if local.shape[-1] < per:
            local = torch.cat([local, torch.zeros(per - local.shape[-1], dtype=local.dtype)], dim=-1)
        parts.append(local)
    return comm.all_gather(parts)[: shape.vocab]


def split_kv_by_rank(K: torch.Tensor, shape: Shape, n: int) -> List[torch.Tensor]:
    """Rank-local view of a global-head cache [nkv, S, hd]: rank r keeps its heads."""
    return [K[kv_heads_of_rank(shape, n, r)].clone() for r in range(n)]


def param_count(shape: Shape, n: int, r: int) -> int:
    """Parameters rank r holds under the shard rules (norms whole on every rank,
    the LM head shared with the embedding when tied)."""
    validate_tp(shape, n)
    H, hd = shape.hidden, shape.head_dim
    per_layer = 0
    full = {"q": (shape.num_q_heads * hd, H), "k": (shape.num_kv_heads * hd, H),
            "v": (shape.num_kv_heads * hd, H), "o": (H, shape.num_q_heads * hd),
            "gate": (shape.intermediate, H), "up": (shape.intermediate, H),
            "down": (H, shape.intermediate)}
    for kind, (rows, cols) in full.items():
        dim, idx = shard_index(kind, shape, n, r)
        per_layer += len(idx) * (cols if dim == "rows" else rows)
    per_layer += 2 * H + 2 * hd
    a, b = vocab_range(shape.vocab, n, r)
    head = (b - a) * H * (1 if shape.tie_word_embeddings else 2) + H
    return shape.num_layers * per_layer + head


# ---------------------------------------------------------------------------
# A step over a batch of sequences (each sequence is independent)
# ---------------------------------------------------------------------------

@dataclasses.dataclass
class SeqInput:
    """One sequence of a step: new-token hidden rows or ids, and per-layer caches
    [nkv, ctx, hd] (global kv heads) of its ctx already-cached positions."""
    hidden: Optional[torch.Tensor]          # [T, H] or None
    ids: Optional[torch.Tensor]             # [T] int64 or None
    k_cache: List[torch.Tensor]
    v_cache: List[torch.Tensor]


@dataclasses.dataclass
class SeqOutput:
    hidden: torch.Tensor                    # [T, H] after the last layer run
    k_cache: List[torch.Tensor]             # extended caches, global heads (as the cache holds them)
    v_cache: List[torch.Tensor]
    logits: Optional[torch.Tensor] = None   # [V] for the last position
    next_id: Optional[int] = None
    k_new: Optional[List[torch.Tensor]] = None  # per layer, the new positions' K / V [nkv, T, hd] before
    v_new: Optional[List[torch.Tensor]] = None  # the cache stored them (unsharded runs)


def run_sequence(seq: SeqInput, layers: Sequence[LayerWeights], hw: Optional[HeadWeights],
                 shape: Shape, n: int = 0, comm: Optional[Comm] = None, head: bool = True,
                 kv_dtype: Optional[torch.dtype] = None) -> SeqOutput:
    """Embedding (if ids) -> layers -> (if hw and head) final norm, logits of the
    last position, argmax.  n == 0 runs unsharded; n >= 1 runs the TP emulation.
    kv_dtype: element type of the KV cache (None: the computing precision)."""
    tp = n >= 1
    if tp:
        validate_tp(shape, n)
        comm = comm if comm is not None else Comm()
    x = seq.hidden
    if seq.ids is not None:
        x = tp_embed(seq.ids, hw, shape, n, comm) if tp else embed(seq.ids, hw)
    ks, vs, k_new, v_new = [], [], [], []
    for li, w in enumerate(layers):
        if tp:
            ranks = [shard_layer(w, shape, n, r) for r in range(n)]
            kc = split_kv_by_rank(seq.k_cache[li], shape, n)
            vc = split_kv_by_rank(seq.v_cache[li], shape, n)
            x, nk, nv = tp_decoder_layer(x, ranks, shape, kc, vc, comm, kv_dtype)
            ks.append(_merge_kv(nk, shape, n))
            vs.append(_merge_kv(nv, shape, n))
        else:
            tr: dict = {}
            x, K, V = decoder_layer(x, w, shape, seq.k_cache[li], seq.v_cache[li], tr, kv_dtype)
            ks.append(K)
            vs.append(V)
            k_new.append(tr["k"])
            v_new.append(tr["v"])
    out = SeqOutput(hidden=x, k_cache=ks, v_cache=vs, k_new=None if tp else k_new, v_new=None if tp else v_new)
    if hw is not None and head:
        logits = tp_lm_head(x[-1], hw, shape, n, comm) if tp else lm_head(x[-1], hw, shape)
        out.logits = logits
        out.next_id = int(argmax_first(logits))
    return out


@dataclasses.dataclass
class SpSeqOutput:
    hidden_chunks: List[torch.Tensor]       # rank r: [token_chunk(T, n, r) rows, H] after the last layer
    k_cache: List[torch.Tensor]             # extended caches, global heads
    v_cache: List[torch.Tensor]
    logits: Optional[torch.Tensor] = None   # [V] for the last position
    next_id: Optional[int] = None


def run_sequence_sp(seq: SeqInput, layers: Sequence[LayerWeights], hw: Optional[HeadWeights], shape: Shape,
                    n: int, comm: Optional[Comm] = None, head: bool = True,
                    kv_dtype: Optional[torch.dtype] = None) -> SpSeqOutput:
    """run_sequence under tensor + sequence parallelism: the residual stream
    lives as token chunks (hidden rows given as input are split the same way)."""
    validate_tp(shape, n)
    comm = comm if comm is not None else Comm()
    if seq.ids is not None:
        x = sp_embed(seq.ids, hw, shape, n, comm)
    else:
        T = seq.hidden.shape[0]
        x = [seq.hidden[slice(*token_chunk(T, n, r))] for r in range(n)]
    ks, vs = [], []
    for li, w in enumerate(layers):
        ranks = [shard_layer(w, shape, n, r) for r in range(n)]
        kc = split_kv_by_rank(seq.k_cache[li], shape, n)
        vc = split_kv_by_rank(seq.v_cache[li], shape, n)
        x, nk, nv = sp_decoder_layer(x, ranks, shape, kc, vc, comm, kv_dtype)
        ks.append(_merge_kv(nk, shape, n))
        vs.append(_merge_kv(nv, shape, n))
    out = SpSeqOutput(hidden_chunks=x, k_cache=ks, v_cache=vs)
    if hw is not None and head:
        out.logits = sp_lm_head(x, hw, shape, n, comm)
        out.next_id = int(argmax_first(out.logits))
    return out


def greedy_generate(prompt: torch.Tensor, layers: Sequence[LayerWeights], hw: HeadWeights, shape: Shape,
                    steps: int, n: int = 0, comm: Optional[Comm] = None,
                    kv_dtype: Optional[torch.dtype] = None) -> Tuple[List[int], List[float], torch.Tensor]:
    """Greedy generation as in "Tensor parallelism from scratch", tp.py main: one
    forward over the prompt with an empty cache, then ``steps`` times: take the
    argmax (first index on ties) of the last position's logits, append it, and run
    a one-token forward that extends the cache.  Returns the chosen ids, the top-2
    margin of the logits each was chosen from, and the logits of the last forward.
    n >= 1 runs every forward through the TP emulation (the page compares the two)."""
    empty = [torch.zeros(shape.num_kv_heads, 0, shape.head_dim, dtype=DTYPE) for _ in layers]
    out = run_sequence(SeqInput(hidden=None, ids=prompt, k_cache=list(empty), v_cache=list(empty)), layers, hw,
                       shape, n=n, comm=comm, kv_dtype=kv_dtype)
    tokens: List[int] = []
    margins: List[float] = []
    for _ in range(steps):
        top2 = torch.topk(out.logits, 2).values
        tokens.append(out.next_id)
        margins.append(float(top2[0] - top2[1]))
        out = run_sequence(SeqInput(hidden=None, ids=torch.tensor([out.next_id]), k_cache=out.k_cache,
                                    v_cache=out.v_cache), layers, hw, shape, n=n, comm=comm, kv_dtype=kv_dtype)
    return tokens, margins, out.logits


def _merge_kv(per_rank: Sequence[torch.Tensor], shape: Shape, n: int) -> torch.Tensor:
    """Global-head cache from rank caches (the first rank holding a head supplies it)."""
    got: Dict[int, torch.Tensor] = {}
    for r in range(n):
        for j, g in enumerate(kv_heads_of_rank(shape, n, r)):
            got.setdefault(g, per_rank[r][j])
    return torch.stack([got[g] for g in range(shape.num_kv_heads)])
