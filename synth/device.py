"""Device half of the seeded generator (``synth/csrc/synth_fill.cu``): fills
torch CUDA buffers with exactly the values ``synth`` draws on the host."""

from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional, Sequence

import torch

import synth

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libtpsynth.so")
_lib = None


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise ImportError(f"{_LIB_PATH} is missing: run __graft_entry__.build() first")
        lib = ctypes.CDLL(_LIB_PATH)
        U64, P, I32, F32 = ctypes.c_uint64, ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        lib.synth_fill_normal_bf16.argtypes = [P, U64, U64, U64, U64, F32, I32, F32, P]
        lib.synth_fill_kv.argtypes = [P, I32, I32, I32, I32, I32, ctypes.POINTER(ctypes.c_int32), I32, U64, U64,
                                      I32, I32, U64, P]
        lib.synth_fill_token_ids.argtypes = [P, U64, U64, U64, U64, U64, P]
        for f in (lib.synth_fill_normal_bf16, lib.synth_fill_kv, lib.synth_fill_token_ids):
            f.restype = ctypes.c_int
        _lib = lib
    return _lib


def _s():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def fill_normal(dst: torch.Tensor, seed: int, stream: int, sigma: float, mean: Optional[float] = None,
                start: int = 0) -> torch.Tensor:
    assert dst.is_cuda and dst.dtype == torch.bfloat16 and dst.is_contiguous()
    rc = _load().synth_fill_normal_bf16(ctypes.c_void_p(dst.data_ptr()), dst.numel(), seed, stream, start,
                                        float(sigma), 0 if mean is None else 1, 0.0 if mean is None else float(mean),
                                        _s())
    if rc:
        raise RuntimeError(f"synth_fill_normal_bf16 failed ({rc})")
    return dst


def token_ids(count: int, vocab: int, seed: int = synth.SEED_TOKENS, stream: int = 0) -> torch.Tensor:
    out = torch.empty(count, dtype=torch.int32, device="cuda")
    rc = _load().synth_fill_token_ids(ctypes.c_void_p(out.data_ptr()), count, vocab, seed, stream, 0, _s())
    if rc:
        raise RuntimeError(f"synth_fill_token_ids failed ({rc})")
    return out


def layer_weights(s: synth.ModelShape, layer: int, perturbed_norms: bool = False) -> Dict[str, torch.Tensor]:
    """Full (unsharded) bf16 tensors of one layer on the device, by name."""
    names = {synth.W_Q: "q", synth.W_K: "k", synth.W_V: "v", synth.W_O: "o", synth.W_GATE: "gate",
             synth.W_UP: "up", synth.W_DOWN: "down", synth.W_IN_NORM: "in_norm", synth.W_POST_NORM: "post_norm",
             synth.W_Q_NORM: "q_norm", synth.W_K_NORM: "k_norm"}
    out = {}
    for kind, shape in synth.layer_weight_shapes(s).items():
        t = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
        if kind in synth.NORM_KINDS:
            if perturbed_norms:
                fill_normal(t, synth.SEED_WEIGHTS, synth.weight_stream(layer, kind), synth.NORM_SIGMA_PERTURBED,
                            mean=1.0)
            else:
                t.fill_(1.0)
        else:
            fill_normal(t, synth.SEED_WEIGHTS, synth.weight_stream(layer, kind), synth.WEIGHT_SIGMA)
        out[names[kind]] = t
    return out


def head_weights(s: synth.ModelShape, perturbed_norms: bool = False) -> Dict[str, torch.Tensor]:
    emb = torch.empty(s.vocab, s.hidden, dtype=torch.bfloat16, device="cuda")
    fill_normal(emb, synth.SEED_WEIGHTS, synth.global_stream(synth.W_EMBED), synth.WEIGHT_SIGMA)
    out = {"embed": emb}
    if not s.tie_word_embeddings:
        lm = torch.empty_like(emb)
        fill_normal(lm, synth.SEED_WEIGHTS, synth.global_stream(synth.W_LM_HEAD), synth.WEIGHT_SIGMA)
        out["lm_head"] = lm
    fn = torch.empty(s.hidden, dtype=torch.bfloat16, device="cuda")
    if perturbed_norms:
        fill_normal(fn, synth.SEED_WEIGHTS, synth.global_stream(synth.W_FINAL_NORM), synth.NORM_SIGMA_PERTURBED,
                    mean=1.0)
    else:
        fn.fill_(1.0)
    out["final_norm"] = fn
    return out


def hidden(num_tokens: int, hidden_size: int) -> torch.Tensor:
    t = torch.empty(num_tokens, hidden_size, dtype=torch.bfloat16, device="cuda")
    return fill_normal(t, synth.SEED_ACTIVATIONS, 0, 1.0)


def fill_kv_cache(cache: torch.Tensor, n: int, max_seqs: int, nkv_l: int, capacity: int, head_dim: int,
                  head_of_local: Sequence[int], num_kv_heads: int, layer: int, num_slots: int, fill_len: int) -> None:
    """Fill positions [0, fill_len) of slots [0, num_slots) of a layer cache laid out
    [n][2][max_seqs][nkv_l][capacity][hd]; head_of_local[r*nkv_l + j] is the global kv
    head stored at rank r's local head j (given by the caller)."""
    m = (ctypes.c_int32 * len(head_of_local))(*head_of_local)
    rc = _load().synth_fill_kv(ctypes.c_void_p(cache.data_ptr()), n, max_seqs, nkv_l, capacity, head_dim, m,
                               num_kv_heads, synth.SEED_KV, layer, num_slots, fill_len, synth.KV_POS_STRIDE, _s())
    if rc:
        raise RuntimeError(f"synth_fill_kv failed ({rc})")
