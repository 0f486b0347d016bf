"""Seeded, counter-based synthetic inputs.

This module is the one piece shared by the CPU oracle and by the GPU tests and
benchmark.  It draws the random weights, activations, KV-cache contents and
token ids that both sides consume, and it holds none of the transformer's
arithmetic: no normalisation, no projection, no sharding rule.

Generator (one definition, implemented here in NumPy and in
``synth/csrc/synth_fill.cu`` for device buffers, bit for bit the same):

* ``mix64`` is the SplitMix64 output function (Steele, Lea and Flood, "Fast
  splittable pseudorandom number generators", OOPSLA 2014; constants as in
  Vigna's public-domain ``splitmix64.c``).
* A (seed, stream) pair selects a key ``key = mix64(seed * G + stream)`` with
  ``G = 0x9E3779B97F4A7C15``; element ``i`` of that stream is
  ``u = mix64(key + (i + 1) * G)`` (all arithmetic mod 2**64).  With key 0 this
  is exactly the SplitMix64 sequence started from state 0.
* An approximately standard normal sample is the Irwin-Hall sum of the four
  16-bit lanes of ``u``: ``x = float32(sum - 131070) * float32(sqrt(3)/65536)``
  (one fp32 multiply, exact operand), then ``y = x * sigma`` (+ ``mean`` in a
  separate fp32 add when a mean is asked for), then round-to-nearest-even to
  bf16.  The sample is bounded by +-3.46 sigma and is never -0.0.
* A token id in ``[0, V)`` is ``((u >> 32) * V) >> 32``.
"""

from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence, Tuple

import numpy as np

GOLDEN = 0x9E3779B97F4A7C15
MIX1 = 0xBF58476D1CE4E5B9
MIX2 = 0x94D049BB133111EB
MASK64 = (1 << 64) - 1
# fp32(sqrt(3) / 65536): scale that gives the 4-lane Irwin-Hall sum unit variance
IH_SCALE = np.float32(np.sqrt(3.0) / 65536.0)
IH_CENTER = 131070  # 4 * (65535 / 2)

# seeds
SEED_WEIGHTS = 0
SEED_ACTIVATIONS = 1
SEED_KV = 2
SEED_TOKENS = 3

# weight stream ids: per layer l the stream is l * 64 + kind; model-wide tensors
# use GLOBAL_STREAM + kind
W_Q, W_K, W_V, W_O, W_GATE, W_UP, W_DOWN, W_IN_NORM, W_POST_NORM, W_Q_NORM, W_K_NORM = range(11)
W_EMBED, W_LM_HEAD, W_FINAL_NORM = range(3)
GLOBAL_STREAM = 1 << 20
KV_POS_STRIDE = 1 << 20  # maximum cached positions per (slot, k|v, head) block


def mix64_int(z: int) -> int:
    """SplitMix64 output function on a Python int (reference for the array form)."""
    z &= MASK64
    z = ((z ^ (z >> 30)) * MIX1) & MASK64
    z = ((z ^ (z >> 27)) * MIX2) & MASK64
    return z ^ (z >> 31)


# Bitwise work goes through the ufuncs explicitly (np.right_shift, ...): on some
# NumPy builds the operator forms (>>, ^, &) on uint64 arrays are far slower.
_RS, _XOR, _AND = np.right_shift, np.bitwise_xor, np.bitwise_and


def _mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output function, in place on a uint64 array (wrapping)."""
    _XOR(z, _RS(z, np.uint64(30)), out=z)
    np.multiply(z, np.uint64(MIX1), out=z)
    _XOR(z, _RS(z, np.uint64(27)), out=z)
    np.multiply(z, np.uint64(MIX2), out=z)
    _XOR(z, _RS(z, np.uint64(31)), out=z)
    return z


def stream_key(seed: int, stream: int) -> int:
    return mix64_int((seed * GOLDEN + stream) & MASK64)


def bits(seed: int, stream: int, index: np.ndarray) -> np.ndarray:
    """Raw 64-bit draws for the given element indices of (seed, stream)."""
    key = np.uint64(stream_key(seed, stream))
    z = np.asarray(index, dtype=np.uint64) + np.uint64(1)
    z *= np.uint64(GOLDEN)
    z += key
    return _mix64(z)


def _f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); inputs here are finite."""
    u = x.astype(np.float32).view(np.uint32)
    rounding = _AND(_RS(u, np.uint32(16)), np.uint32(1)) + np.uint32(0x7FFF)
    return _RS(u + rounding, np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return np.left_shift(np.asarray(b, dtype=np.uint16).astype(np.uint32), np.uint32(16)).view(np.float32)


def normal_bf16_bits_at(seed: int, stream: int, index: np.ndarray, sigma: float,
                        mean: Optional[float] = None) -> np.ndarray:
    """bf16 bit patterns of the approximately N(mean, sigma^2) draws at ``index``."""
    u = bits(seed, stream, index)
    m = np.uint64(0xFFFF)
    s = _AND(u, m)
    s += _AND(_RS(u, np.uint64(16)), m)
    s += _AND(_RS(u, np.uint64(32)), m)
    s += _RS(u, np.uint64(48))
    x = (s.astype(np.int64) - IH_CENTER).astype(np.float32) * IH_SCALE
    y = x * np.float32(sigma)
    if mean is not None:
        y = y + np.float32(mean)
    return _f32_to_bf16_bits(y)


def normal_bf16_bits(seed: int, stream: int, count: int, sigma: float,
                     mean: Optional[float] = None, start: int = 0,
                     chunk: int = 1 << 20) -> np.ndarray:
    """``count`` consecutive draws of a stream, as bf16 bit patterns (uint16)."""
    out = np.empty(count, dtype=np.uint16)
    for c0 in range(0, count, chunk):
        c1 = min(count, c0 + chunk)
        idx = np.arange(start + c0, start + c1, dtype=np.uint64)
        out[c0:c1] = normal_bf16_bits_at(seed, stream, idx, sigma, mean)
    return out


def token_ids(seed: int, stream: int, count: int, vocab: int, start: int = 0) -> np.ndarray:
    """Token ids uniform in ``[0, vocab)`` (int64)."""
    u = bits(seed, stream, np.arange(start, start + count, dtype=np.uint64))
    return _RS(_RS(u, np.uint64(32)) * np.uint64(vocab), np.uint64(32)).astype(np.int64)


# ---------------------------------------------------------------------------
# Workloads: shapes, batch structure and the seeds/streams of every input.
# ---------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class ModelShape:
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


@dataclasses.dataclass(frozen=True)
class Workload:
    """One step: ``prefill`` sequences (q_len, cached ctx) then ``decode`` sequences."""
    name: str
    shape: ModelShape
    tp_sizes: Tuple[int, ...]
    prefill: Tuple[Tuple[int, int], ...]   # (q_len, ctx_len) per prefill sequence
    decode: Tuple[int, ...]                # ctx_len per decode sequence (q_len == 1)
    layers_run: int                        # decoder layers in one step
    input_from_ids: bool                   # step starts at the embedding (else hidden ~N(0,1))

    @property
    def num_seqs(self) -> int:
        return len(self.prefill) + len(self.decode)

    @property
    def q_lens(self) -> List[int]:
        return [q for q, _ in self.prefill] + [1] * len(self.decode)

    @property
    def ctx_lens(self) -> List[int]:
        return [c for _, c in self.prefill] + list(self.decode)

    @property
    def num_tokens(self) -> int:
        return sum(self.q_lens)


QWEN3_06B = ModelShape(hidden=1024, num_q_heads=16, num_kv_heads=8, head_dim=128,
                       intermediate=3072, vocab=151936, num_layers=28, tie_word_embeddings=True)
QWEN3_32B = ModelShape(hidden=5120, num_q_heads=64, num_kv_heads=8, head_dim=128,
                       intermediate=25600, vocab=151936, num_layers=64, tie_word_embeddings=False)
TINY = ModelShape(hidden=256, num_q_heads=4, num_kv_heads=2, head_dim=64,
                  intermediate=768, vocab=1024, num_layers=1, tie_word_embeddings=True)

WORKLOADS = {
    # tiny layer + vocab head, tp 2, prefill 8 tokens from ids
    "tiny_prefill8": Workload("tiny_prefill8", TINY, (2,), ((8, 0),), (), 1, True),
    # one 0.6B-shaped layer, prefill 1 x 2048 tokens, hidden ~N(0,1)
    "qwen3_0.6b_layer_prefill2048": Workload("qwen3_0.6b_layer_prefill2048", QWEN3_06B, (1, 2),
                                             ((2048, 0),), (), 1, False),
    # one 0.6B-shaped layer, decode 64 seqs x 1 token over 4096 cached tokens, + LM head
    "qwen3_0.6b_layer_decode64x4096": Workload("qwen3_0.6b_layer_decode64x4096", QWEN3_06B, (1, 2, 4),
                                               (), (4096,) * 64, 1, False),
    # one 32B-shaped layer at tp 16 (KV heads replicated on 2 ranks)
    "qwen3_32b_layer_tp16_decode32x2048": Workload("qwen3_32b_layer_tp16_decode32x2048", QWEN3_32B, (16,),
                                                   (), (2048,) * 32, 1, False),
    "qwen3_32b_layer_tp16_prefill1024": Workload("qwen3_32b_layer_tp16_prefill1024", QWEN3_32B, (16,),
                                                 ((1024, 0),), (), 1, False),
    # full 28-layer 0.6B model, mixed step: 4 x 512 prefill + 128 decode at ctx 2048
    "qwen3_0.6b_model_mixed": Workload("qwen3_0.6b_model_mixed", QWEN3_06B, (1, 2, 4),
                                       ((512, 0),) * 4, (2048,) * 128, 28, True),
}


def weight_stream(layer: int, kind: int) -> int:
    return layer * 64 + kind


def global_stream(kind: int) -> int:
    return GLOBAL_STREAM + kind


def layer_weight_shapes(s: ModelShape) -> dict:
    """[out, in] shapes of one decoder layer's full (unsharded) tensors."""
    H, hd = s.hidden, s.head_dim
    return {
        W_Q: (s.num_q_heads * hd, H),
        W_K: (s.num_kv_heads * hd, H),
        W_V: (s.num_kv_heads * hd, H),
        W_O: (H, s.num_q_heads * hd),
        W_GATE: (s.intermediate, H),
        W_UP: (s.intermediate, H),
        W_DOWN: (H, s.intermediate),
        W_IN_NORM: (H,),
        W_POST_NORM: (H,),
        W_Q_NORM: (hd,),
        W_K_NORM: (hd,),
    }


NORM_KINDS = (W_IN_NORM, W_POST_NORM, W_Q_NORM, W_K_NORM)
WEIGHT_SIGMA = 0.02
NORM_SIGMA_PERTURBED = 0.1


def layer_weight_bits(s: ModelShape, layer: int, kind: int, perturbed_norms: bool = False) -> np.ndarray:
    """bf16 bits of one full layer tensor (norm weights are 1, or 1 + N(0, 0.1))."""
    shape = layer_weight_shapes(s)[kind]
    count = int(np.prod(shape))
    if kind in NORM_KINDS:
        if not perturbed_norms:
            return np.full(shape, 0x3F80, dtype=np.uint16)
        return normal_bf16_bits(SEED_WEIGHTS, weight_stream(layer, kind), count,
                                NORM_SIGMA_PERTURBED, mean=1.0).reshape(shape)
    return normal_bf16_bits(SEED_WEIGHTS, weight_stream(layer, kind), count, WEIGHT_SIGMA).reshape(shape)


def global_weight_bits(s: ModelShape, kind: int, perturbed_norms: bool = False) -> np.ndarray:
    if kind == W_FINAL_NORM:
        if not perturbed_norms:
            return np.full((s.hidden,), 0x3F80, dtype=np.uint16)
        return normal_bf16_bits(SEED_WEIGHTS, global_stream(kind), s.hidden,
                                NORM_SIGMA_PERTURBED, mean=1.0)
    count = s.vocab * s.hidden
    return normal_bf16_bits(SEED_WEIGHTS, global_stream(kind), count, WEIGHT_SIGMA).reshape(s.vocab, s.hidden)


def hidden_bits(num_tokens: int, hidden: int, start_token: int = 0) -> np.ndarray:
    """Input hidden states ~N(0,1) for single-layer workloads, rows = packed tokens."""
    return normal_bf16_bits(SEED_ACTIVATIONS, 0, num_tokens * hidden, 1.0,
                            start=start_token * hidden).reshape(num_tokens, hidden)


def step_token_ids(num_tokens: int, vocab: int) -> np.ndarray:
    return token_ids(SEED_TOKENS, 0, num_tokens, vocab)


def kv_cache_index(slot: int, kv: int, head: int, pos: np.ndarray, num_kv_heads: int, head_dim: int) -> np.ndarray:
    """Counter index of cached element (slot, k=0|v=1, global kv head, pos, :)."""
    base = ((slot * 2 + kv) * num_kv_heads + head) * KV_POS_STRIDE
    pos = np.asarray(pos, dtype=np.uint64)
    return (np.uint64(base) + pos)[..., None] * np.uint64(head_dim) + np.arange(head_dim, dtype=np.uint64)


def kv_cache_bits(layer: int, slot: int, kv: int, head: int, length: int,
                  num_kv_heads: int, head_dim: int) -> np.ndarray:
    """[length, head_dim] bf16 bits of the synthetic cached K (kv=0) or V (kv=1)."""
    idx = kv_cache_index(slot, kv, head, np.arange(length), num_kv_heads, head_dim)
    return normal_bf16_bits_at(SEED_KV, layer, idx.reshape(-1), 1.0).reshape(length, head_dim)
