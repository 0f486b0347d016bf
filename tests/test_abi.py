"""The C-ABI library without a GPU: it loads, exports every declared entry
point, validates shard rules, and its host index maps equal the oracle's."""

import os
import re

import numpy as np
import pytest

import synth
from oracle import forward as of
from oracle import inputs as oi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    text = open(os.path.join(ROOT, "include", "tpfwd.h")).read()
    return sorted(set(re.findall(r"^(?:tp_status|const char\*)\s+(tp_\w+)\s*\(", text, re.M)))


def test_library_exports_every_declared_symbol():
    from tensor_transformer_forward_gb300 import binding
    lib = binding.lib()
    names = _declared()
    assert len(names) >= 17
    for name in names:
        assert hasattr(lib, name), name
    assert sorted(binding.EXPORTED) == names


def _cfg(s: synth.ModelShape, n: int):
    from tensor_transformer_forward_gb300 import ModelConfig
    return ModelConfig(s.hidden, s.num_q_heads, s.num_kv_heads, s.head_dim, s.intermediate, s.vocab, s.num_layers,
                       s.rms_eps, s.rope_theta, n, s.tie_word_embeddings)


CASES = [(synth.TINY, 2), (synth.QWEN3_06B, 1), (synth.QWEN3_06B, 2), (synth.QWEN3_06B, 4),
         (synth.QWEN3_06B, 8), (synth.QWEN3_32B, 16), (synth.QWEN3_32B, 8),
         (synth.ModelShape(hidden=128, num_q_heads=8, num_kv_heads=2, head_dim=64, intermediate=96, vocab=1000,
                           num_layers=1), 4)]


@pytest.mark.parametrize("s,n", CASES)
def test_index_maps_match_oracle_bit_exactly(s, n):
    from tensor_transformer_forward_gb300 import Context
    ctx = Context(_cfg(s, n))
    shape = oi.shape_of(s)
    for r in range(n):
        for kind in ("q", "k", "v", "o", "gate", "up", "down", "embed", "lm_head"):
            dim, idx = ctx.shard_index_map(kind, r)
            odim, oidx = of.shard_index(kind, shape, n, r)
            assert dim == odim and np.array_equal(np.asarray(idx, dtype=np.int64), oidx), (kind, r)


def test_uneven_vocab_slices_and_replicated_heads():
    from tensor_transformer_forward_gb300 import Context
    s = synth.ModelShape(hidden=128, num_q_heads=8, num_kv_heads=2, head_dim=64, intermediate=96, vocab=1000,
                         num_layers=1)
    ctx = Context(_cfg(s, 3 if False else 4))
    lens = [len(ctx.shard_index_map("embed", r)[1]) for r in range(4)]
    assert lens == [250, 250, 250, 250]
    s3 = synth.ModelShape(hidden=128, num_q_heads=6, num_kv_heads=3, head_dim=64, intermediate=96, vocab=1000,
                          num_layers=1)
    ctx3 = Context(_cfg(s3, 3))
    assert [len(ctx3.shard_index_map("embed", r)[1]) for r in range(3)] == [334, 334, 332]
    heads = [ctx.shard_index_map("k", r)[1][0] // 64 for r in range(4)]
    assert heads == [0, 0, 1, 1]


@pytest.mark.parametrize("kw,code", [
    (dict(num_q_heads=28, num_kv_heads=4), "TP_ERR_HEADS_NOT_DIVISIBLE"),
    (dict(num_q_heads=24, num_kv_heads=12), "TP_ERR_KV_HEADS"),
    (dict(num_q_heads=16, num_kv_heads=2, intermediate=100), "TP_ERR_INTERMEDIATE"),
    (dict(vocab=13), "TP_ERR_VOCAB"),
    (dict(head_dim=96), "TP_ERR_UNSUPPORTED"),
])
def test_create_rejects_what_the_pages_rule_out(kw, code):
    import tensor_transformer_forward_gb300 as tpf
    base = dict(hidden=256, num_q_heads=16, num_kv_heads=8, head_dim=64, intermediate=256, vocab=1000, num_layers=1)
    base.update(kw)
    s = synth.ModelShape(**base)
    with pytest.raises(tpf.TPError) as e:
        tpf.Context(_cfg(s, 8))
    assert e.value.status == getattr(tpf, code)
    # the oracle rejects the same shards (kernel coverage aside)
    if code != "TP_ERR_UNSUPPORTED":
        with pytest.raises(of.ShardError):
            of.validate_tp(oi.shape_of(s), 8)


def test_layout_sizes():
    from tensor_transformer_forward_gb300 import WEIGHTS_HEAD, WEIGHTS_LAYER, Context
    s, n = synth.QWEN3_32B, 16
    ctx = Context(_cfg(s, n))
    H, hd = s.hidden, s.head_dim
    off, nb = ctx.weights_part("qkv")
    assert nb == n * (4 + 2) * hd * H * 2          # 4 q heads + replicated k and v head per rank
    assert ctx.weights_part("gate_up")[1] == n * 2 * 1600 * H * 2
    assert ctx.weights_part("down")[1] == n * H * 1600 * 2
    assert ctx.weights_part("lm_head")[0] != ctx.weights_part("embed")[0]  # untied
    assert ctx.weights_bytes(WEIGHTS_LAYER) >= sum(ctx.weights_part(p)[1] for p in ("qkv", "o", "gate_up", "down"))
    assert ctx.kv_cache_bytes(32, 2112) == n * 2 * 32 * 1 * 2112 * hd * 2
    t = Context(_cfg(synth.QWEN3_06B, 2))
    assert t.weights_part("lm_head")[0] != t.weights_part("embed")[0]       # fp16 operand copy even when tied
    assert t.rank_sum_count() == 0


def test_binding_refuses_pageable_host_buffers():
    """ids / out_ids may be CUDA tensors or page-locked CPU tensors (read and written
    by the kernels over the host link); other CPU memory is refused before any call."""
    import torch
    from tensor_transformer_forward_gb300 import binding
    with pytest.raises(ValueError, match="page-locked"):
        binding._dev_or_pinned(torch.zeros(4, dtype=torch.int32), "ids", torch.int32)
    with pytest.raises(ValueError):
        binding._dev(torch.zeros(4, dtype=torch.int32), "ids", torch.int32)


def test_entry_points_refuse_empty_or_missing_inputs_before_device_work():
    """Degenerate calls (no tokens, no sequences, no workspace, null buffers) come back
    as TP_ERR_INVALID_ARG from host-side checks, with nothing launched."""
    import ctypes
    from tensor_transformer_forward_gb300 import Context, binding
    L = binding._lib
    ctx = Context(_cfg(synth.TINY, 2))
    h = ctx.handle
    fake = ctypes.c_void_p(4096)  # never dereferenced: every call below fails its checks first
    inval = binding.TP_ERR_INVALID_ARG
    assert L.tp_embed_vocab_parallel(h, fake, fake, 0, fake, fake, None) == inval          # no tokens
    assert L.tp_embed_vocab_parallel(h, fake, None, 4, fake, fake, None) == inval          # no ids
    b = binding.TPBatch()
    b.num_seqs, b.num_tokens = 0, 0
    assert L.tp_decoder_layer_forward(h, fake, ctypes.byref(b), fake, fake, 1, 64, fake, None) == inval  # no workspace
    assert L.tp_lm_head_argmax(h, fake, ctypes.byref(b), fake, fake, None, fake, None) == inval
    assert L.tp_decoder_layer_forward(None, fake, ctypes.byref(b), fake, fake, 1, 64, fake, None) == inval
    nb = ctypes.c_size_t()
    assert L.tp_kv_cache_bytes(h, 0, 64, ctypes.byref(nb)) == inval                         # no sequences
    assert L.tp_kv_cache_bytes(h, 1, 0, ctypes.byref(nb)) == inval                          # no positions
    assert L.tp_hidden_written(None) == inval
    assert ctx.launch_count() == 0


def test_static_scratch_entry_point_refuses_sizes_beyond_its_array_before_device_work():
    """tp_lm_head_argmax_static has a fixed scratch array: more than 64 sequences or a
    hidden size above 8192 comes back as TP_ERR_INVALID_ARG from the host-side checks,
    before any CUDA call (this runs without a GPU)."""
    import ctypes
    from tensor_transformer_forward_gb300 import Context, binding
    L = binding._lib
    fake = ctypes.c_void_p(4096)  # never dereferenced: the size checks come first
    inval = binding.TP_ERR_INVALID_ARG
    big = synth.ModelShape(hidden=8256, num_q_heads=16, num_kv_heads=8, head_dim=128, intermediate=256,
                           vocab=1024, num_layers=1)
    ctx = Context(_cfg(big, 1))
    b = binding.TPBatch()
    b.num_seqs, b.num_prefill, b.num_tokens, b.max_q_len, b.max_kv_len = 1, 0, 1, 1, 1
    b.cu_q = b.ctx_len = b.slot = 4096
    assert L.tp_lm_head_argmax_static(ctx.handle, fake, ctypes.byref(b), fake, fake, None, fake, None) == inval
    small = Context(_cfg(synth.TINY, 2))
    b.num_seqs, b.num_tokens = 65, 65
    assert L.tp_lm_head_argmax_static(small.handle, fake, ctypes.byref(b), fake, fake, None, fake, None) == inval
    assert ctx.launch_count() == 0 and small.launch_count() == 0


@pytest.mark.parametrize("s,n", [(synth.TINY, 2), (synth.QWEN3_06B, 1), (synth.QWEN3_06B, 2), (synth.QWEN3_32B, 16)])
def test_workspace_holds_the_declared_intermediates_and_grows_with_its_limits(s, n):
    """tp_workspace_bytes against what the header says the workspace holds: the
    four per-token intermediates (fp16 layer output [T, H], the merged projection
    [T, n, (nq_l + 2 nkv_l) hd] in 16-bit, the attention output [T, n nq_l hd] and
    SiLU * up [T, n I_p] in fp16) and the fp32 RoPE (cos, sin) table of every
    position; never smaller when a limit grows, and by at least the per-token
    parts for every further 128-token tile and by about the table's rows for
    more positions (regions are padded)."""
    from tensor_transformer_forward_gb300 import Context
    ctx = Context(_cfg(s, n))
    nq_l, nkv_l, hd = s.num_q_heads // n, max(1, s.num_kv_heads // n), s.head_dim
    per_token = 2 * s.hidden + 2 * n * (nq_l + 2 * nkv_l) * hd + 2 * n * nq_l * hd + 2 * n * (s.intermediate // n)
    for T, S, P in [(1, 1, 1), (64, 64, 4097), (2048, 1, 2049), (2176, 132, 2049)]:
        b = ctx.workspace_bytes(T, S, P)
        assert b >= T * per_token + P * hd * 4, (T, S, P, b)
        assert ctx.workspace_bytes(2 * T, S, P) >= b
        if T % 128 == 0:
            assert ctx.workspace_bytes(2 * T, S, P) - b >= T * per_token
        assert ctx.workspace_bytes(T, 2 * S, P) >= b
        assert ctx.workspace_bytes(T, S, 2 * P) >= b
        if P >= 1024:  # the table is padded too: allow up to 128 positions of it
            assert ctx.workspace_bytes(T, S, 2 * P) - b >= (P - 128) * hd * 4
